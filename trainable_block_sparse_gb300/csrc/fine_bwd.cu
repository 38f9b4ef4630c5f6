// Fine stage of VSA, backward (the method trains end to end: "VSA: Faster
// Video Diffusion with Trainable Sparse Attention", abstract; gradients of the
// masked fine attention of App. B with the selection held fixed):
//   P  = exp(S * scale - lse)           (recomputed from the saved log-sum-exp)
//   dP = dO_f V^T,  dS = P (.) (dP - delta),  delta = rowsum(dO_f (.) O_f)
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO_f
// over the selected 64x64 blocks only.  The pooled (coarse) gradients enter
// as dQ += repeat(dQ_c)/64 etc. in the epilogue, which also un-permutes.
// dO_f and delta arrive multiplied by a power of two per (batch, head) slice
// (the combine backward's gradient scale, which keeps small upstream gradients
// inside fp16's normal range); dP, dS, dQ, dK and dV are linear in them, so the
// epilogue divides the accumulators by the slice's factor (exactly).
//
// One tcgen05 kernel template runs two deterministic, atomic-free passes:
//  * kKeyMajor = false (dQ pass): work item = two query cubes (M = 128 query
//    rows), walking the union of their index lists.  X1 = Q, X2 = dO_f of the
//    item; per step of two key cubes Y1 = K, Y2 = V:
//    S = Q K^T, dP = dO V^T, the softmax warps turn them into dS, dQ += dS K.
//  * kKeyMajor = true (dK/dV pass): work item = two key cubes (M = 128 key
//    rows), walking the union of their transposed lists (query cubes that
//    selected them).  X1 = K, X2 = V; per step of two query cubes Y1 = Q,
//    Y2 = dO: S^T = K Q^T, dP^T = V dO^T, the softmax warps write P^T and dS^T
//    (fp16) into the dP columns, then dV += P^T dO and dK += dS^T Q.
// Operands are the fp16 staged copies of Q, K, V and dO_f; P and dS are fp16.
//
// Per step the softmax warps signal twice: once S has been read (so the next
// step's S product can be issued at once) and once dS is in TMEM.  TMEM
// (512 columns): S at 0, dP at 128, the dQ or dV accumulator at 256; at 384
// the dK accumulator (key-major pass) or, in the dQ pass, the item's Q and
// dO as TMEM A operands (D/2 columns each), copied from X by the softmax
// warps, so the S and dP products read only K and V from shared memory.  In
// the dQ pass dS(t) is packed over the dP columns, so dP(t+1) is issued after
// dQ(t) has read them.
// Y1 and Y2 come through separate TMA rings (Y1 is read by the last product
// of a step, Y2 earlier, so Y1 gets the deeper ring).
// Epilogue: four epilogue warps (one per TMEM lane quarter) read the
// accumulators out of TMEM, scale them, add the pooled gradient and write them
// (fp32, or rounded once to bf16 if the caller asks for bf16 gradients)
// straight to global memory, four threads per row and 32 whole bytes of a row
// per group, while the softmax warps go on with the next item (a 128 KB drain
// takes several thousand cycles at the SM's store rate, so it must not hold
// them).  dQ pass: X(i+1) is loaded once Q and dO of item i are in TMEM, and
// the next item's first dQ product waits until the epilogue has read dQ.
// Key-major pass: the next item's K and V are loaded as soon as the item's
// last S^T and dP^T products are done; its first dV product waits until the
// epilogue has read dV, its first dK product until it has read dK.
// Warps 0-7: softmax; warp w reads TMEM lane quarter w%4 (32 rows) and the 64
// columns of step tile w/4, so each thread owns half a row.  Warp 8: TMA loads
// of Y1/Y2.  Warp 9: UMMA issue.  Warp 10: TMA loads of X.  Warp 11: item
// fetcher (the next item from the launch's shared counter, item_seq.cuh).
// Warps 12-15: epilogue.  Registers are split per warpgroup: 168 a thread for
// the softmax warps, 88 for the rest.
// Bounded waits and the abort path are as in the forward kernel.
#include "item_seq.cuh"
#include "umma_pipe.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreadsBwd = 512;  // 16 warps
constexpr int kSoftmaxWarpsBwd = 8;
constexpr int kWarpLoadY = 8, kWarpIssue = 9, kWarpLoadX = 10, kWarpEpi0 = 12;  // 11: fetcher
constexpr int kEpiWarps = 4;
// readers of the item sequence: Y and X producer threads, UMMA warp, softmax
// and epilogue warps
constexpr int kSeqReadersBwd = 3 + kSoftmaxWarpsBwd + kEpiWarps;
// register split: the launch gives 65536 / 512 = 128 a thread
constexpr int kRegsSoftmax = 168, kRegsRest = 88;
static_assert(256 * kRegsSoftmax + 256 * kRegsRest <= 65536, "split exceeds the launch's registers");
// setmaxnreg.inc only raises and .dec only lowers a warp's count (the launch
// gives 128): a .dec above the launch's count is an illegal instruction.
static_assert(kRegsSoftmax >= 128 && kRegsRest <= 128 && kRegsSoftmax % 8 == 0 &&
                  kRegsRest % 8 == 0 && kRegsRest >= 24,
              "setmaxnreg shares must move away from the launch's count, in steps of 8");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColA1 = 256, kColA2 = 384;
// dQ pass: the item's Q and dO as TMEM A operands (D/2 columns each) at kColA2
constexpr float kLog2e = 1.4426950408889634f;
template <int D>
struct BwdSmem {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;          // 128 rows x 128 bytes
  static constexpr int kXBytes = kChunks * kChunkBytes;  // one 128-row operand
  static constexpr int kStages1 = (D == 128) ? 3 : 4;    // Y1 ring
  static constexpr int kStages2 = (D == 128) ? 2 : 4;    // Y2 ring
  static constexpr int kTileBytes = 64 * D * 2;
  static constexpr int kBytes = (2 + kStages1 + kStages2) * kXBytes + 1024;
};

struct BwdBars {
  uint64_t x_full;
  uint64_t y1_full[4], y1_empty[4], y2_full[4], y2_empty[4];
  uint64_t s_full, s_read, dp_full[2], ds_full[2];  // dP/dS barriers by step parity
  uint64_t acc_full, acc_free, final_mma;  // acc_free: dQ pass, the epilogue has read dQ
  uint64_t a_ready, x_free;  // dQ pass: the item's Q, dO copied from X into TMEM
  uint64_t x_empty;          // key-major pass: the item's last S^T and dP^T are done
  uint64_t dv_free, dk_free; // key-major pass: the epilogue has read dV / dK
  ItemSeq seq;
  uint32_t tmem_base;
  int abort;
};

struct BwdParams {
  Geom g;
  const PairItem* items;
  const uint32_t* lists;
  int n_items;
  const int* order;       // schedule position -> item (null: identity)
  const float* lse;     // [BH, N] cube order, natural log
  const float* delta;   // [BH, N] cube order
  const float* gscale;  // [BH] factor dO_f and delta carry (null: 1)
  const float* pooled1; // dQ_c (dQ pass) or dV_c (key-major pass), may be null
  const float* pooled2; // dK_c (key-major pass), may be null
  void* out1;           // dQ (dQ pass) or dV (key-major pass), caller layout, fp32 or
                        // bf16 (g.grad_bf16)
  void* out2;           // dK (key-major pass)
  uint32_t* status;
  int* sched;           // schedule counter, zero at launch
};

__device__ __forceinline__ void warp_arrive_bwd(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Two gradient values to out[i], out[i + 1] (8 bytes fp32, or 4 bytes bf16
// rounded to nearest even).
template <class T>
__device__ __forceinline__ void store2(T* out, size_t i, float x, float y) {
  if constexpr (std::is_same<T, float>::value)
    *reinterpret_cast<float2*>(out + i) = make_float2(x, y);
  else
    *reinterpret_cast<__nv_bfloat162*>(out + i) = __floats2bfloat162_rn(x, y);
}

// Columns [c0, c0 + D/2) of one output row of an item with no selected
// blocks: only pooled[cube]/64 reaches it (plain stores; a rare path).
template <int D, class T>
__device__ __forceinline__ void store_pooled_half(int c0, const float* pooled, size_t pooled_row,
                                                  T* out, size_t out_row) {
#pragma unroll 1
  for (int cc = c0; cc < c0 + D / 2; cc += 2) {
    float2 r = make_float2(0.f, 0.f);
    if (pooled) {
      const float2 a = *reinterpret_cast<const float2*>(pooled + pooled_row * D + cc);
      r = make_float2(a.x * (1.f / kTile), a.y * (1.f / kTile));
    }
    store2(out, out_row * D + cc, r.x, r.y);
  }
}

template <int D>
__device__ __forceinline__ void store_pooled_half(bool bf16, int c0, const float* pooled,
                                                  size_t pooled_row, void* out, size_t out_row) {
  if (bf16)
    store_pooled_half<D>(c0, pooled, pooled_row, static_cast<__nv_bfloat16*>(out), out_row);
  else
    store_pooled_half<D>(c0, pooled, pooled_row, static_cast<float*>(out), out_row);
}

// Key-major epilogue: the 32 accumulator rows of this warp's lane quarter
// (at TMEM address tq), times `mul` plus the pooled gradient, to global
// memory; row 16h + 8j + t/4 of the quarter goes to output row orow[2h + j].
// pp[k] holds, in lane l, pooled columns 2(l + 32k) and 2(l + 32k) + 1,
// already divided by 64.
template <int D, class T>
__device__ __forceinline__ void drain_acc(uint32_t tq, float mul, const float2 (&pp)[D / 64],
                                          T* out, const size_t (&orow)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[2][16];
    tmem_ld16x256_x4(tq + 32 * c, v[0]);
    tmem_ld16x256_x4(tq + (16u << 16) + 32 * c, v[1]);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // column pair 16c + 4i + t%4 sits in lane (that) % 32 of pp[c / 2]
      const int src = 16 * (c & 1) + 4 * i + (lane & 3);
      const float px = __shfl_sync(0xffffffffu, pp[c >> 1].x, src);
      const float py = __shfl_sync(0xffffffffu, pp[c >> 1].y, src);
      const int col = 32 * c + 8 * i + 2 * (lane & 3);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j)
          store2(out, orow[2 * h + j] * D + col,
                 fmaf(__uint_as_float(v[h][4 * i + 2 * j]), mul, px),
                 fmaf(__uint_as_float(v[h][4 * i + 2 * j + 1]), mul, py));
    }
  }
}

template <int D>
__device__ __forceinline__ void drain_acc(bool bf16, uint32_t tq, float mul,
                                          const float2 (&pp)[D / 64], void* out,
                                          const size_t (&orow)[4]) {
  if (bf16)
    drain_acc<D>(tq, mul, pp, static_cast<__nv_bfloat16*>(out), orow);
  else
    drain_acc<D>(tq, mul, pp, static_cast<float*>(out), orow);
}

template <int D, bool kKeyMajor>
__global__ void __launch_bounds__(kThreadsBwd, 1)
    fine_bwd_kernel(const __grid_constant__ CUtensorMap tx1, const __grid_constant__ CUtensorMap tx2,
                    const __grid_constant__ CUtensorMap ty1, const __grid_constant__ CUtensorMap ty2,
                    BwdParams P) {
  using L = BwdSmem<D>;
  constexpr int kS1 = L::kStages1, kS2 = L::kStages2;
  constexpr int kKSteps = D / 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sX1 = smem;
  uint8_t* sX2 = sX1 + L::kXBytes;
  uint8_t* sY1 = sX2 + L::kXBytes;  // ring of kS1 operands
  uint8_t* sY2 = sY1 + kS1 * L::kXBytes;
  __shared__ BwdBars sb;
  int* abort_flag = &sb.abort;
  const Geom& g = P.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&sb.x_full, 1);
    for (int i = 0; i < kS1; ++i) {
      mbar_init(&sb.y1_full[i], 1);
      mbar_init(&sb.y1_empty[i], 1);
    }
    for (int i = 0; i < kS2; ++i) {
      mbar_init(&sb.y2_full[i], 1);
      mbar_init(&sb.y2_empty[i], 1);
    }
    mbar_init(&sb.s_full, 1);
    mbar_init(&sb.s_read, kSoftmaxWarpsBwd);   // one arrival per softmax warp
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.dp_full[i], 1);
      mbar_init(&sb.ds_full[i], kSoftmaxWarpsBwd);
    }
    mbar_init(&sb.acc_full, 1);
    mbar_init(&sb.acc_free, kEpiWarps);
    mbar_init(&sb.a_ready, kSoftmaxWarpsBwd);
    mbar_init(&sb.x_free, kSoftmaxWarpsBwd);
    mbar_init(&sb.x_empty, 1);
    mbar_init(&sb.dv_free, kEpiWarps);
    mbar_init(&sb.dk_free, kEpiWarps);
    mbar_init(&sb.final_mma, 1);
    seq_init(sb.seq, kSeqReadersBwd);
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
  // dP buffer of global step t (one buffer: the dQ pass keeps Q and dO in TMEM)
  auto dpcol = [](uint32_t) -> uint32_t { return kColDP; };
  constexpr uint32_t kColQT = kColA2, kColDOT = kColA2 + D / 2;  // dQ pass

  if (warp == kWarpLoadY) {
    // ===================================================== TMA loads of Y1, Y2
    regs_dec<kRegsRest>();
    if (lane == 0) {
      tma_prefetch_desc(&ty1);
      tma_prefetch_desc(&ty2);
      uint32_t n1 = 0, n2 = 0;  // steps whose Y1 / Y2 copies were issued
      uint32_t sq = 0;
      bool ok = true;
      while (ok) {
        const int item = seq_next<false>(sb.seq, sq, abort_flag, P.status);
        if (item < 0 || is_aborted(abort_flag)) break;
        const PairItem pi = P.items[P.order ? P.order[item] : item];
        if (pi.count == 0) continue;
        const uint32_t* list = P.lists + pi.off;
        const int nsteps = (pi.count + 1) / 2;
        for (int s = 0; s < nsteps; ++s) {
          const uint32_t step = n1;
          const bool two = 2 * s + 1 < pi.count;
          const int t0 = static_cast<int>(list[2 * s] & 0xFFFFu);
          const int t1 = two ? static_cast<int>(list[2 * s + 1] & 0xFFFFu) : t0;
          const int r0 = pi.bh * g.N + t0 * kTile, r1 = pi.bh * g.N + t1 * kTile;
          const uint32_t bytes = (two ? 2 : 1) * L::kTileBytes;
          const uint32_t sl1 = step % kS1, sl2 = step % kS2;
          if (step >= static_cast<uint32_t>(kS1) &&
              !wait1(&sb.y1_empty[sl1], ((step / kS1) & 1) ^ 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          uint8_t* y1 = sY1 + sl1 * L::kXBytes;
          mbar_arrive_expect_tx(&sb.y1_full[sl1], bytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_2d(y1 + c * L::kChunkBytes, &ty1, c * 64, r0, &sb.y1_full[sl1]);
            if (two) tma_load_2d(y1 + c * L::kChunkBytes + 8192, &ty1, c * 64, r1, &sb.y1_full[sl1]);
          }
          ++n1;
          if (step >= static_cast<uint32_t>(kS2) &&
              !wait1(&sb.y2_empty[sl2], ((step / kS2) & 1) ^ 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          uint8_t* y2 = sY2 + sl2 * L::kXBytes;
          mbar_arrive_expect_tx(&sb.y2_full[sl2], bytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_2d(y2 + c * L::kChunkBytes, &ty2, c * 64, r0, &sb.y2_full[sl2]);
            if (two) tma_load_2d(y2 + c * L::kChunkBytes + 8192, &ty2, c * 64, r1, &sb.y2_full[sl2]);
          }
          ++n2;
        }
      }
      // Drain: every copy issued must land before the CTA can exit (slots
      // older than one ring length were already waited for before reuse).
      for (uint32_t t = n1 > static_cast<uint32_t>(kS1) ? n1 - kS1 : 0; t < n1; ++t)
        mbar_wait(&sb.y1_full[t % kS1], (t / kS1) & 1, kWaitNs);
      for (uint32_t t = n2 > static_cast<uint32_t>(kS2) ? n2 - kS2 : 0; t < n2; ++t)
        mbar_wait(&sb.y2_full[t % kS2], (t / kS2) & 1, kWaitNs);
    }
  } else if (warp == kWarpIssue) {
    // ===================================================== UMMA issuer
    regs_dec<kRegsRest>();
    const uint32_t id_s128 = idesc_f16(128, 128, 0, 0);
    const uint32_t id_s64 = idesc_f16(128, 64, 0, 0);
    const uint32_t id_acc = idesc_f16(128, D, 0, 1);
    const uint64_t x1d0 = sdesc_sw128(smem_u32(sX1), 16, 1024);
    const uint64_t x2d0 = sdesc_sw128(smem_u32(sX2), 16, 1024);
    const uint64_t y1k0 = sdesc_sw128(smem_u32(sY1), 16, 1024);              // K-major views
    const uint64_t y2k0 = sdesc_sw128(smem_u32(sY2), 16, 1024);
    const uint64_t y1m0 = sdesc_sw128(smem_u32(sY1), L::kChunkBytes, 1024);  // MN-major views
    const uint64_t y2m0 = sdesc_sw128(smem_u32(sY2), L::kChunkBytes, 1024);
    uint64_t x1d[kKSteps], x2d[kKSteps];
#pragma unroll
    for (int k = 0; k < kKSteps; ++k) {
      const uint32_t o = ((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4;
      x1d[k] = x1d0 + o;
      x2d[k] = x2d0 + o;
    }
    auto kdesc = [&](uint64_t base, uint32_t slot, uint64_t (&yd)[kKSteps]) {
      const uint32_t off = (slot * L::kXBytes) >> 4;
#pragma unroll
      for (int k = 0; k < kKSteps; ++k)
        yd[k] = base + off + (((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);
    };
    // A (TMEM, packed fp16 pairs, D/2 columns) x B^T (K-major smem): D/16 MMAs
    auto issue_ts_chain = [&](uint32_t d, uint32_t a, const uint64_t (&b)[kKSteps],
                              uint32_t ids) {
      issue_ts4(d, a, b[0], b[1], b[2], b[3], ids, 0u);
      if constexpr (kKSteps == 8) issue_ts4(d, a + 32, b[4], b[5], b[6], b[7], ids, 1u);
    };
    // S (or S^T) of global step t: X1 x Y1^T (dQ pass: X1 = Q from TMEM)
    auto issue_s = [&](uint32_t t, uint32_t ids) -> bool {
      const uint32_t sl = t % kS1;
      if (!waitw(&sb.y1_full[sl], (t / kS1) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      uint64_t yd[kKSteps];
      kdesc(y1k0, sl, yd);
      if (kKeyMajor) issue_ss_chain<kKSteps>(tb + kColS, x1d, yd, ids);
      else issue_ts_chain(tb + kColS, tb + kColQT, yd, ids);
      commit_elect(&sb.s_full);
      return true;
    };
    // dP (or dP^T) of global step t: X2 x Y2^T (dQ pass: X2 = dO from TMEM)
    auto issue_dp = [&](uint32_t t, uint32_t ids) -> bool {
      const uint32_t sl = t % kS2;
      if (!waitw(&sb.y2_full[sl], (t / kS2) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      uint64_t yd[kKSteps];
      kdesc(y2k0, sl, yd);
      if (kKeyMajor) issue_ss_chain<kKSteps>(tb + dpcol(t), x2d, yd, ids);
      else issue_ts_chain(tb + dpcol(t), tb + kColDOT, yd, ids);
      commit_elect(&sb.dp_full[t & 1]);
      if (!kKeyMajor) commit_elect(&sb.y2_empty[sl]);  // V feeds only dP in the dQ pass
      return true;
    };
    uint32_t step = 0;  // global index of the current item's first step
    uint32_t sq = 0;
    int it = 0;
    bool ok = true;
    while (ok) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (item < 0 || is_aborted(abort_flag)) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;
      const int nsteps = (pi.count + 1) / 2;
      // key-major: X1 = K, X2 = V in shared memory; dQ pass: Q, dO in TMEM
      if (!waitw(kKeyMajor ? &sb.x_full : &sb.a_ready, it & 1, abort_flag, P.status)) break;
      const uint32_t ids0 = pi.count > 1 ? id_s128 : id_s64;
      if (!issue_s(step, ids0) || !issue_dp(step, ids0)) break;
      for (int s = 0; s < nsteps; ++s) {
        const uint32_t t = step + s;
        const bool two = 2 * s + 1 < pi.count;
        const bool more = s + 1 < nsteps;
        const uint32_t nids = (2 * s + 3 < pi.count) ? id_s128 : id_s64;
        const uint32_t sl1 = t % kS1, sl2 = t % kS2;
        // key-major: every S^T and dP^T product of the item has been issued;
        // X (K and V of the item) is free once they are done
        if (kKeyMajor && !more) commit_elect(&sb.x_empty);
        // softmax phase 1 of step t is done: S(t) has been read (and, in the
        // key-major pass, replaced by P^T)
        if ((kKeyMajor || more) && !waitw(&sb.s_read, t & 1, abort_flag, P.status)) {
          ok = false;
          break;
        }
        if (kKeyMajor) {
          if (s == 0 && it > 0 && !waitw(&sb.dv_free, (it - 1) & 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dV += P^T dO   (P^T packed in the S columns, dO = Y2)
          issue_ts_rows(tb + kColA1, tb + kColS, y2m0 + ((sl2 * L::kXBytes) >> 4), two, id_acc,
                        s > 0, 64);
          commit_elect(&sb.y2_empty[sl2]);
        }
        if (more) {
          // S(t+1) overwrites S(t) (or P^T(t), after dV(t) has read it)
          if (!issue_s(t + 1, nids)) { ok = false; break; }
        }
        if (!waitw(&sb.ds_full[t & 1], (t >> 1) & 1, abort_flag, P.status)) { ok = false; break; }
        if (s == 0 && it > 0 &&
            !waitw(kKeyMajor ? &sb.dk_free : &sb.acc_free, (it - 1) & 1, abort_flag, P.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!kKeyMajor) {
          // dQ += dS K   (dS packed in dP buffer t, K = Y1 as an MN-major operand)
          issue_ts_rows(tb + kColA1, tb + dpcol(t), y1m0 + ((sl1 * L::kXBytes) >> 4), two, id_acc,
                        s > 0, 64);
          commit_elect(&sb.y1_empty[sl1]);
          // dP(t+1) overwrites the dP columns after dQ(t) has read them
          if (more && !issue_dp(t + 1, nids)) { ok = false; break; }
        } else {
          // dK += dS^T Q   (dS^T packed in the dP columns, Q = Y1)
          issue_ts_rows(tb + kColA2, tb + kColDP, y1m0 + ((sl1 * L::kXBytes) >> 4), two, id_acc,
                        s > 0, 64);
          commit_elect(&sb.y1_empty[sl1]);
          // dP(t+1) overwrites the dP columns after dK(t) has read them
          if (more && !issue_dp(t + 1, nids)) { ok = false; break; }
        }
      }
      if (!ok) break;
      commit_elect(&sb.acc_full);
      step += nsteps;
      ++it;
    }
    commit_elect(&sb.final_mma);
    mbar_wait(&sb.final_mma, 0, kWaitNs);
  } else if (warp == kWarpLoadX) {
    // ===================================================== TMA loads of X
    regs_dec<kRegsRest>();
    if (lane == 0) {
      tma_prefetch_desc(&tx1);
      tma_prefetch_desc(&tx2);
      // X1 (h = 0) or X2 (h = 1) of item pi
      auto load_x = [&](const PairItem& pi, int h) {
        const CUtensorMap* m = h ? &tx2 : &tx1;
        uint8_t* dst = h ? sX2 : sX1;
        const int ra = pi.bh * g.N + pi.a * kTile;
        const int rb = pi.bh * g.N + (pi.b >= 0 ? pi.b : pi.a) * kTile;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_2d(dst + c * L::kChunkBytes, m, c * 64, ra, &sb.x_full);
          tma_load_2d(dst + c * L::kChunkBytes + 8192, m, c * 64, rb, &sb.x_full);
        }
      };
      int it = 0;
      uint32_t sq = 0;
      for (;;) {
        const int item = seq_next<false>(sb.seq, sq, abort_flag, P.status);
        if (item < 0 || is_aborted(abort_flag)) break;
        const PairItem pi = P.items[P.order ? P.order[item] : item];
        if (pi.count == 0) continue;
        // X of the previous item is no longer read: key-major, its last S^T
        // and dP^T products are done; dQ pass, its Q and dO are in TMEM
        if (it > 0 && !wait1(kKeyMajor ? &sb.x_empty : &sb.x_free, (it - 1) & 1, abort_flag,
                             P.status))
          break;
        mbar_arrive_expect_tx(&sb.x_full, 2 * L::kXBytes);
        load_x(pi, 0);
        load_x(pi, 1);
        ++it;
      }
      if (it > 0) mbar_wait(&sb.x_full, (it - 1) & 1, kWaitNs);  // the last copy lands
    }
  } else if (warp < kSoftmaxWarpsBwd) {
    // ===================================================== softmax-backward
    regs_inc<kRegsSoftmax>();
    const int quarter = warp & 3;
    const int hc = warp >> 2;                 // step tile = column half of S and dP
    const int row = quarter * 32 + lane;
    const int half = row >> 6;                // warp-uniform: the item cube of these rows
    const uint32_t mybit = half ? kSelB : kSelA;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = g.scale * kLog2e;
    const uint32_t ts = tb + lane_addr + kColS + 64 * hc;
    constexpr uint32_t kFull = 0xffffffffu;
    uint32_t step = 0;
    int it = 0;
    bool ok = true;
    // dQ pass: copies this thread's half row of Q (X1) and dO (X2) of the item
    // whose operands are in X into the TMEM A-operand columns, then signals
    // the UMMA warp (a_ready) and the X producer (x_free).
    auto copy_x_to_tmem = [&](int ix) -> bool {
      if (!waitw(&sb.x_full, ix & 1, abort_flag, P.status)) return false;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint8_t* base = m ? sX2 : sX1;
        uint32_t w[D / 4];
#pragma unroll
        for (int u = 0; u < D / 16; ++u) {
          const int chunk = D == 128 ? hc : 0, unit = D == 128 ? u : 4 * hc + u;
          const uint4 v = *reinterpret_cast<const uint4*>(
              base + chunk * L::kChunkBytes + row * 128 + ((unit ^ (row & 7)) << 4));
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
        const uint32_t col = tb + lane_addr + (m ? kColDOT : kColQT) + (D / 4) * hc;
        if constexpr (D == 128) tmem_st32(col, w);
        else tmem_st16(col, w);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive_bwd(&sb.a_ready);
      warp_arrive_bwd(&sb.x_free);
      return true;
    };
    uint32_t sq = 0;
    bool x_in_tmem = false;  // dQ pass: this item's Q and dO are already in TMEM
    // dQ pass: the next item's row lse and delta, loaded while this item runs
    int pre_item = kSeqEnd;
    float pre_lse = 0.f, pre_delta = 0.f;
    while (ok) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (item < 0 || is_aborted(abort_flag)) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      const int cube = half ? pi.b : pi.a;
      const bool row_live = half == 0 || pi.b >= 0;
      const size_t prow = static_cast<size_t>(pi.bh) * g.Nc + cube;
      if (pi.count == 0) {
        // no fine contribution: only the pooled gradient reaches these rows
        if (row_live) {
          const size_t orow = static_cast<size_t>(pi.bh) * g.N + caller_row(g, cube, row & 63);
          store_pooled_half<D>(g.grad_bf16, hc * (D / 2), P.pooled1, prow, P.out1, orow);
          if (kKeyMajor)
            store_pooled_half<D>(g.grad_bf16, hc * (D / 2), P.pooled2, prow, P.out2, orow);
        }
        continue;
      }
      const uint32_t* list = P.lists + pi.off;
      // dQ pass: an item's Q and dO go to TMEM at the end of the item before it
      // (below), or here if that item did not see it coming
      if (!kKeyMajor && !x_in_tmem && !copy_x_to_tmem(it)) break;
      x_in_tmem = false;
      float row_lse = 0.f, row_delta = 0.f;
      if (!kKeyMajor && row_live) {
        if (item == pre_item) {
          row_lse = pre_lse * kLog2e;
          row_delta = pre_delta;
        } else {
          const size_t frow = static_cast<size_t>(pi.bh) * g.N + cube * kTile + (row & 63);
          row_lse = P.lse[frow] * kLog2e;
          row_delta = P.delta[frow];
        }
      }
      if (!kKeyMajor) {
        // the next item's lse and delta of this row: the loads are issued now
        // and first used when that item starts
        const int nx = seq_peek(sb.seq, sq, 0, abort_flag, P.status);
        if (nx == kSeqAbort) break;
        pre_item = nx;
        if (nx >= 0) {
          const PairItem pn = P.items[P.order ? P.order[nx] : nx];
          if (pn.count > 0 && (half == 0 || pn.b >= 0)) {
            const size_t nrow =
                static_cast<size_t>(pn.bh) * g.N + (half ? pn.b : pn.a) * kTile + (row & 63);
            pre_lse = P.lse[nrow];
            pre_delta = P.delta[nrow];
          }
        }
      }
      const int nsteps = (pi.count + 1) / 2;
      // key-major: lse (log2 units) and delta of the step tile's 64 query rows,
      // lane l holding rows l and 32 + l, broadcast with shuffles; fetched one
      // step ahead (the loads' values are first touched, lse scaled to log2
      // units, when the step they belong to begins).  (Warp-uniform 16-byte
      // loads from L1 instead of the shuffles measured 13% slower on the 720p
      // layer.)
      auto tile_rows = [&](int s2, float& l0, float& l1, float& d0, float& d1) {
        const bool h2 = hc == 0 || 2 * s2 + 1 < pi.count;
        const uint32_t e2 = h2 ? list[2 * s2 + hc] : 0u;
        const size_t q0 = static_cast<size_t>(pi.bh) * g.N + (e2 & 0xFFFFu) * kTile;
        l0 = __ldg(P.lse + q0 + lane);
        l1 = __ldg(P.lse + q0 + 32 + lane);
        d0 = __ldg(P.delta + q0 + lane);
        d1 = __ldg(P.delta + q0 + 32 + lane);
      };
      float cl0 = 0.f, cl1 = 0.f, cd0 = 0.f, cd1 = 0.f;
      if (kKeyMajor) {
        tile_rows(0, cl0, cl1, cd0, cd1);
        cl0 *= kLog2e;
        cl1 *= kLog2e;
      }
      // list entry of this half's step tile, fetched one step ahead
      uint32_t e_cur = hc < pi.count ? __ldg(list + hc) : 0u;
      for (int s = 0; s < nsteps; ++s, ++step) {
        const bool two = 2 * s + 1 < pi.count;
        const bool have = hc == 0 || two;   // this step has a tile for this column half
        const bool valid = have && (e_cur & mybit) != 0;  // warp-uniform
        e_cur = __ldg(list + min(2 * s + 2 + hc, pi.count - 1));  // in bounds; unused past the list
        float nl0 = 0.f, nl1 = 0.f, nd0 = 0.f, nd1 = 0.f;
        if (kKeyMajor && s + 1 < nsteps) tile_rows(s + 1, nl0, nl1, nd0, nd1);
        if (!waitw(&sb.s_full, step & 1, abort_flag, P.status)) { ok = false; break; }
        tc_fence_after();
        // ---- phase 1: P from S (key-major: P^T packed over the S columns)
        float p[64];
        if (valid) {
          unroll_for<2>([&](auto CH) {
            constexpr int ch = decltype(CH)::value;
            uint32_t sv[32];
            tmem_ld32(ts + 32 * ch, sv);
            tmem_wait_ld();
            // scale-and-shift on fp32 pairs
            unroll_for<16>([&](auto J) {
              constexpr int j = 2 * decltype(J)::value;
              const float l0 = kKeyMajor ? __shfl_sync(kFull, ch ? cl1 : cl0, j) : row_lse;
              const float l1 = kKeyMajor ? __shfl_sync(kFull, ch ? cl1 : cl0, j + 1) : row_lse;
              float t0, t1;
              fma2(t0, t1, __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]), c, c, -l0, -l1);
              p[32 * ch + j] = ex2_approx(t0);
              p[32 * ch + j + 1] = ex2_approx(t1);
            });
          });
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) p[j] = 0.f;
        }
        if (kKeyMajor && have) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_f16x2(p[2 * i], p[2 * i + 1]);
          tmem_st32(ts, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        warp_arrive_bwd(&sb.s_read);
        // ---- phase 2: dS = P (.) (dP - delta)
        const uint32_t b = step & 1;
        if (!waitw(&sb.dp_full[b], (step >> 1) & 1, abort_flag, P.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tdp = tb + lane_addr + dpcol(step) + 64 * hc;
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
                const int j = 2 * i;
                const float dl0 = kKeyMajor ? __shfl_sync(kFull, ch ? cd1 : cd0, j) : row_delta;
                const float dl1 = kKeyMajor ? __shfl_sync(kFull, ch ? cd1 : cd0, j + 1) : row_delta;
                float d0, d1;
                submul2(d0, d1, __uint_as_float(dv[j]), __uint_as_float(dv[j + 1]), dl0, dl1,
                        p[32 * ch + j], p[32 * ch + j + 1]);
                dk[i] = pack_f16x2(d0, d1);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) dk[i] = 0u;
            }
            // chunk ch packs into 16 columns at 16*ch (columns already read)
            tmem_st16(tdp + 16 * ch, dk);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        warp_arrive_bwd(&sb.ds_full[b]);
        cl0 = nl0 * kLog2e;
        cl1 = nl1 * kLog2e;
        cd0 = nd0;
        cd1 = nd1;
      }
      if (!ok) break;
      if (!kKeyMajor) {
        // every S and dP product of this item is complete (phase 2 of its last
        // step saw its dP): the next item's Q and dO may replace these in TMEM,
        // so its first products run while the epilogue warps drain dQ.  The
        // next item with work is looked up in the sequence without reading
        // it off, a few entries ahead at most.
        int nx = kSeqEnd;
        for (int a = 0; a <= kSeqSlots - 2; ++a) {
          const int p = seq_peek(sb.seq, sq, a, abort_flag, P.status);
          if (p < 0 || P.items[P.order ? P.order[p] : p].count > 0) {
            nx = p;
            break;
          }
        }
        if (nx == kSeqAbort) break;
        if (nx >= 0) {
          if (!copy_x_to_tmem(it + 1)) break;
          x_in_tmem = true;
        }
      }
      ++it;
    }
  } else if (warp >= kWarpEpi0) {
    // ===================================================== epilogue
    regs_dec<kRegsRest>();
    const int quarter = warp & 3;
    const bool second = quarter >= 2;  // rows 64..127: the item's second cube
    const uint32_t tq = tb + (static_cast<uint32_t>(quarter * 32) << 16);
    int it = 0;
    uint32_t sq = 0;
    for (;;) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (item < 0 || is_aborted(abort_flag)) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;  // the softmax warps write its pooled rows
      const int cube = second ? pi.b : pi.a;
      const bool live = !second || pi.b >= 0;  // warp-uniform
      size_t orow[4];
      float2 p1[D / 64], p2[D / 64];
#pragma unroll
      for (int k = 0; k < D / 64; ++k) p1[k] = p2[k] = make_float2(0.f, 0.f);
      if (live) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
          orow[r] = static_cast<size_t>(pi.bh) * g.N +
                    caller_row(g, cube, (32 * quarter + 8 * r + lane / 4) & 63);
        const size_t prow = static_cast<size_t>(pi.bh) * g.Nc + cube;
#pragma unroll
        for (int k = 0; k < D / 64; ++k) {
          const size_t o = prow * D + 2 * (lane + 32 * k);
          if (P.pooled1) {
            const float2 a = __ldg(reinterpret_cast<const float2*>(P.pooled1 + o));
            p1[k] = make_float2(a.x * (1.f / kTile), a.y * (1.f / kTile));
          }
          if (P.pooled2) {
            const float2 a = __ldg(reinterpret_cast<const float2*>(P.pooled2 + o));
            p2[k] = make_float2(a.x * (1.f / kTile), a.y * (1.f / kTile));
          }
        }
      }
      // 1 / (the slice's gradient scale): a power of two, so exact
      const float inv_gs = P.gscale ? 1.f / __ldg(P.gscale + pi.bh) : 1.f;
      if (!waitw(&sb.acc_full, it & 1, abort_flag, P.status)) break;
      tc_fence_after();
      // dQ pass: dQ = scale * acc; key-major: dV = acc, then dK = scale * acc
      // (each divided by the gradient scale)
      if (live)
        drain_acc<D>(g.grad_bf16, tq + kColA1, (kKeyMajor ? 1.f : g.scale) * inv_gs, p1, P.out1,
                     orow);
      tc_fence_before();
      warp_arrive_bwd(kKeyMajor ? &sb.dv_free : &sb.acc_free);
      if (kKeyMajor) {
        if (live) drain_acc<D>(g.grad_bf16, tq + kColA2, g.scale * inv_gs, p2, P.out2, orow);
        tc_fence_before();
        warp_arrive_bwd(&sb.dk_free);
      }
      ++it;
    }
  } else {
    // ===================================================== item fetcher
    // (warp 11; its register share completes warpgroup 2's split)
    regs_dec<kRegsRest>();
    if (lane == 0) seq_fetch(sb.seq, P.sched, P.n_items, abort_flag, P.status);
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
  // the register split assumes the launch's 128 registers a thread: setmaxnreg
  // raises the softmax warps above it and lowers the others below it
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs < kRegsRest || attr.numRegs > kRegsSoftmax ||
      attr.numRegs * kThreadsBwd < 256 * (kRegsSoftmax + kRegsRest))
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(p.n_items);
  if (grid <= 0) return cudaSuccess;
  if ((e = cudaMemsetAsync(p.sched, 0, sizeof(int), s)) != cudaSuccess) return e;
  kern<<<grid, kThreadsBwd, smem, s>>>(m1, m2, m3, m4, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_impl(const Geom& g, const __half* q, const __half* k, const __half* v,
                     const float* lse_f, const __half* dof, const float* delta,
                     const float* gscale, const float* dqc, const float* dkc, const float* dvc,
                     void* dq, void* dk, void* dv, const Workspace& ws, cudaStream_t s) {
  const bool ordered = use_cost_order(g);
  BwdParams pq{g, ws.qpairs, ws.qlist, ws.n_qpairs, ordered ? ws.qorder : nullptr, lse_f, delta,
               gscale, dqc, nullptr, dq, nullptr, ws.status, ws.counter + kCounterBwdQ};
  cudaError_t e = run_bwd<D, false>(g, q, dof, k, v, pq, s);
  if (e != cudaSuccess) return e;
  BwdParams pk{g, ws.kpairs, ws.klist, ws.n_kpairs, ordered ? ws.korder : nullptr, lse_f, delta,
               gscale, dvc, dkc, dv, dk, ws.status, ws.counter + kCounterBwdK};
  return run_bwd<D, true>(g, k, v, q, dof, pk, s);
}

}  // namespace

cudaError_t launch_fine_bwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                            const float* lse_f, const __half* dof, const float* delta,
                            const float* gscale, const float* dqc, const float* dkc,
                            const float* dvc, void* dq, void* dk, void* dv,
                            const Workspace& ws, cudaStream_t s) {
  if (g.D == 64)
    return bwd_impl<64>(g, q, k, v, lse_f, dof, delta, gscale, dqc, dkc, dvc, dq, dk, dv, ws, s);
  return bwd_impl<128>(g, q, k, v, lse_f, dof, delta, gscale, dqc, dkc, dvc, dq, dk, dv, ws, s);
}

}  // namespace vsa

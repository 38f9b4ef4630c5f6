// Fine stage of VSA, forward, fused with the gated combine ("VSA: Faster Video
// Diffusion with Trainable Sparse Attention", §2 "Fine stage" and App. B:
// token-level attention only inside the selected 64x64 blocks; paper notes
// 关键设计 3: O = O_c (.) G_c + O_f (.) G_f).
//
// Head_dim 128 (head_dim 64 runs in fine_fwd64.cu, two CTAs per SM).
// GB300 design (tcgen05 + TMEM + TMA, one persistent CTA per SM):
//  * Work item = two query cubes of one (batch, head): their 2 x 64 token rows
//    form one M = 128 tensor-core tile, and the item walks the union of the two
//    index lists (list entries carry which cube selected the key cube; rows of
//    the other cube treat that block as masked).
//  * Steps take two key cubes at a time, so S = Q K^T is an M=128, N=128 UMMA
//    chain and O += P V an M=128, N=D, K=128 chain (N=64 UMMAs run at ~60% of
//    the tensor pipe, N=128 at ~97%).
//  * Q, K, V arrive as fp16 cube-order staged copies and P is written in fp16:
//    with the running maximum kept stale (below), the largest P entries are
//    rounded too, and fp16's 11-bit significand keeps that error 8x below
//    bf16's.  Every UMMA is fp16 x fp16 with fp32 accumulation.
//  * Sixteen warps:
//      warps 0-7   softmax: warp w reads TMEM lane quarter w%4 (32 token rows)
//                  and key tile w/4 of the step (64 columns), so each thread
//                  owns half a row; the two halves of a row agree on the
//                  running maximum through shared memory once per step, and
//                  P goes back into TMEM as the A operand of the PV product;
//      warps 8-11  epilogue: normalise O_f, apply the gates with the cube's
//                  coarse output, write O (bf16, caller layout, un-permuted on
//                  the way out), O_f (fp16, kept for the backward) and the
//                  log-sum-exp;
//      warp 12     TMA: Q once per item, then K tiles gathered by list entry;
//      warp 13     UMMA issue (whole warp converged, one elected lane);
//      warp 14     TMA: V tiles gathered by list entry;
//      warp 15     item fetcher: takes the CTA's next item from the launch's
//                  shared counter and hands it to the other roles
//                  (item_seq.cuh), so the CTAs finish within about an item.
//  * TMEM (512 columns): two S buffers (128 columns each) and two O
//    accumulators.  P(t) (fp16 pairs, 64 columns) is written over the first
//    columns of S(t)'s buffer once both warps of a row pair have read their
//    halves of S(t).  QK^T of step t+1 goes to the other buffer right after
//    PV(t-1) is issued, without waiting for S(t) to be read; the product that
//    next writes a buffer, S(t+2), is issued after PV(t), which reads P(t)
//    there, and the products run in issue order (as the backward's dP(t+1)
//    after dQ(t)).  One full barrier per S buffer for S and one for P.  The
//    epilogue of item i drains one O accumulator while item i+1 accumulates
//    into the other.
//  * The running maximum is only moved (and O rescaled in TMEM) when it grows
//    by more than 2^8, which keeps exp arguments bounded and the rescale rare.
// Every mbarrier wait is bounded; a time-out is recorded in the status word and
// the CTA unwinds, waits for its own in-flight copies and MMAs, frees TMEM and
// exits.
//
// bf16 variant (inference: no O_f): Q, K, V are read in place from the caller's
// bf16 tensors, P is written as bf16 and the UMMAs are kind::f16 with bf16
// operands.  In raster layout every 64-token tile is fetched as one 5-D TMA box
// (64 channels x 4 x 4 x 4 tokens of a [BH, T, H, W, D] view), which lands in
// shared memory in the in-cube token order: the permute happens inside the
// copy and no staged copy is made.
//
// e4m3 variant (kF8, head_dim 128, inference: no O_f): Q, K and V arrive as the
// e4m3 copies of stage_fp8.cu (per-slice power-of-two factors), P is written
// to TMEM as e4m3 and every UMMA is kind::f8f6f4 (K = 32 per MMA) with fp32
// accumulation.  A K tile is 64 rows of 128 bytes (one 128-byte swizzle
// chunk); V comes transposed per cube (64-byte rows of keys, 64-byte swizzle),
// so the P V product reads it K-major.  The per-slice factors of Q and K fold
// into the softmax scale, that of V into the epilogue's normalisation.  Same
// roles, rings, barriers and schedule as the fp16 kernel, half the bytes per
// step.
#include <cfloat>
#include <cstring>

#include "item_seq.cuh"
#include "umma_pipe.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreadsFwd = 512;           // 16 warps
constexpr int kSoftmaxWarps = 8, kEpiWarps = 4;
constexpr int kWarpEpi = 8, kWarpK = 12, kWarpMma = 13, kWarpV = 14, kWarpSeq = 15;
// readers of the item sequence: K and V producer threads, UMMA warp, softmax
// and epilogue warps
constexpr int kSeqReaders = 3 + kSoftmaxWarps + kEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;              // two S buffers of 128 columns (P over S)
constexpr uint32_t kColO = 256;            // O accumulators at columns 256 and 384
constexpr float kRescaleThreshold = 8.0f;  // log2 units (P stays within [0, 256])
// Operand kinds of the kernel: the fp16 staged copies, the e4m3 copies, or the
// caller's bf16 tensors read in place.
enum : int { kOpF16 = 0, kOpE4M3 = 1, kOpBF16 = 2 };
template <int D, bool kF8 = false>
struct FwdSmem {
  // 128-byte chunks of a row: 64 fp16 columns, or 128 e4m3 columns
  static constexpr int kChunks = kF8 ? D / 128 : D / 64;
  static constexpr int kChunkBytes = 128 * 128;       // one chunk of 128 rows
  static constexpr int kQBytes = kChunks * kChunkBytes;
  static constexpr int kKVBytes = kChunks * kChunkBytes;  // 2 key tiles
  static constexpr int kStagesK = kF8 ? 3 : 2;
  // Two stages each.  Deeper rings measured slower: TMA serves a CTA's copies
  // in order, so every extra slot in flight queues ahead of the tile the next
  // product needs (2 K / 3 V and 3 K / 2 V both lost ~1%).  The e4m3 tiles are
  // half as large.
  static constexpr int kStagesV = kF8 ? 3 : 2;
  static constexpr int kTileBytes = 64 * D * (kF8 ? 1 : 2);  // one 64-row tile
  // epilogue staging of one 32-column chunk of O_f: 128 rows x 128 bytes
  static constexpr int kStageOff = kQBytes + (kStagesK + kStagesV) * kKVBytes;
  static constexpr int kStageBytes = 128 * 128;
  static constexpr int kBytes = kStageOff + kStageBytes + 1024;
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[6], k_empty[6], v_full[6], v_empty[6];
  uint64_t s_full[2], p_full[2];  // by step parity = S buffer (P is written over S)
  uint64_t o_full[2], o_free[2];
  uint64_t st_full[2], st_free[2];
  uint64_t final_mma;
  ItemSeq seq;
  uint32_t tmem_base;
  int abort;
  float red[2][2][128];    // [step parity][row half]: the half-row maxima of a step
  float l_part[2][2][128]; // [O buffer][row half]: partial running sums
  float m_fin[2][128];     // [O buffer]: final running maximum (log2 units)
};

struct FwdParams {
  Geom g;
  const PairItem* items;
  const uint32_t* lists;
  int n_items;
  const int* order;       // schedule position -> item (null: identity)
  const __nv_bfloat16* gc;
  const __nv_bfloat16* gf;
  const float* oc;
  __nv_bfloat16* o;
  __half* o_f;
  float* lse_f;
  uint32_t* status;
  const float* scales;    // e4m3 variant: [BH][3] factors of the Q, K, V copies
  int* sched;             // schedule counter, zero at launch
};

// Arrival of a whole warp counted once: lanes finish their own work first.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Named barrier over the four epilogue warps, returning the OR of `fail`
// over them (the warps leave an item loop together; see pair_sync_or).
__device__ __forceinline__ bool epi_sync_or(bool fail) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 5, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(fail))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 5, 128;" ::: "memory"); }

// Named barrier over the two softmax warps that share a TMEM lane quarter,
// returning the OR of `fail` over both warps, so the pair always takes the
// same branch after it (a warp that left alone would strand its partner at the
// next barrier, which has no time limit).
__device__ __forceinline__ bool pair_sync_or(int quarter, bool fail) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(fail)), "r"(1 + quarter)
      : "memory");
  return r != 0;
}

template <int D, int kOp>
__global__ void __launch_bounds__(kThreadsFwd, 1)
    fine_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tof,
                    FwdParams P) {
  constexpr bool kF8 = kOp == kOpE4M3, kBF = kOp == kOpBF16;
  static_assert(!kF8 || D == 128, "the e4m3 variant is for head_dim 128");
  using L = FwdSmem<D, kF8>;
  constexpr int kSK = L::kStagesK, kSV = L::kStagesV;
  constexpr int kKSteps = kF8 ? D / 32 : D / 16;  // K per MMA: 32 e4m3 or 16 fp16 (32 bytes)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + L::kQBytes;
  uint8_t* sV = sK + kSK * L::kKVBytes;
  uint8_t* sStage = smem + L::kStageOff;  // epilogue staging of O_f
  __shared__ FwdBars sb;
  int* abort_flag = &sb.abort;

  const Geom& g = P.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&sb.q_full, 1);
    mbar_init(&sb.q_empty, 1);
    for (int i = 0; i < kSK; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
    }
    for (int i = 0; i < kSV; ++i) {
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.p_full[i], kSoftmaxWarps);  // one arrival per softmax warp
      mbar_init(&sb.o_full[i], 1);
      mbar_init(&sb.o_free[i], kEpiWarps);      // one arrival per epilogue warp
      mbar_init(&sb.st_full[i], kSoftmaxWarps);
      mbar_init(&sb.st_free[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sb.s_full[i], 1);
    mbar_init(&sb.final_mma, 1);
    seq_init(sb.seq, kSeqReaders);
    sb.abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sb.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = sb.tmem_base;

  if (warp == kWarpK || warp == kWarpV) {
    // ===================================================== TMA producers
    // One warp loads Q (once per item) and the K tiles, another the V tiles,
    // each through its own ring, so K for step t is fetched as soon as QK^T of
    // step t - kSK has consumed its slot, independently of the PV products.
    const bool is_k = warp == kWarpK;
    if (lane == 0) {
      const CUtensorMap* tmap = is_k ? &tk : &tv;
      uint64_t* full = is_k ? sb.k_full : sb.v_full;
      uint64_t* empty = is_k ? sb.k_empty : sb.v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const uint32_t kS = is_k ? kSK : kSV;
      tma_prefetch_desc(tmap);
      if (is_k) tma_prefetch_desc(&tq);
      // one 64-row tile (64 columns of it) of a cube of slice bh: a 2-D box of a
      // cube-order tensor, or (bf16 variant, raster layout) a 5-D box of the
      // caller's raster tensor
      auto load_tile = [&](uint8_t* dst, const CUtensorMap* m, int c, int bh, int cube,
                           uint64_t* bar) {
        if (kBF && g.raster) {
          const int cw_ = cube % g.cw, rest = cube / g.cw;
          tma_load_5d(dst, m, c * 64, 4 * cw_, 4 * (rest % g.ch), 4 * (rest / g.ch), bh, bar);
        } else {
          tma_load_2d(dst, m, c * 64, bh * g.N + cube * kTile, bar);
        }
      };
      uint32_t step = 0, sq = 0;
      int it = 0;  // items with work seen by this CTA
      for (;;) {
        const int item = seq_next<false>(sb.seq, sq, abort_flag, P.status);
        if (item < 0 || is_aborted(abort_flag)) break;
        const PairItem pi = P.items[P.order ? P.order[item] : item];
        if (pi.count == 0) continue;
        const uint32_t* list = P.lists + pi.off;
        if (is_k) {
          if (it > 0 && !wait1(&sb.q_empty, (it - 1) & 1, abort_flag, P.status)) break;
          mbar_arrive_expect_tx(&sb.q_full, L::kQBytes);
          const int cube_b = pi.b >= 0 ? pi.b : pi.a;
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            load_tile(sQ + c * L::kChunkBytes, &tq, c, pi.bh, pi.a, &sb.q_full);
            load_tile(sQ + c * L::kChunkBytes + 8192, &tq, c, pi.bh, cube_b, &sb.q_full);
          }
        }
        ++it;
        const int nsteps = (pi.count + 1) / 2;
        bool ok = true;
        for (int s = 0; s < nsteps; ++s) {
          const uint32_t slot = step % kS, ph = (step / kS) & 1;
          const bool two = 2 * s + 1 < pi.count;
          const int t0 = static_cast<int>(list[2 * s] & 0xFFFFu);
          const int t1 = two ? static_cast<int>(list[2 * s + 1] & 0xFFFFu) : t0;
          if (step >= kS &&
              !wait1(&empty[slot], ph ^ 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          uint8_t* dst = ring + slot * L::kKVBytes;
          mbar_arrive_expect_tx(&full[slot], (two ? 2 : 1) * L::kTileBytes);
          if (kF8 && !is_k) {
            // transposed V: rows (cube, channel) of 64 key bytes, one box per cube
            const int v0 = (pi.bh * g.Nc + t0) * D, v1 = (pi.bh * g.Nc + t1) * D;
            tma_load_2d(dst, tmap, 0, v0, &full[slot]);
            if (two) tma_load_2d(dst + 8192, tmap, 0, v1, &full[slot]);
          } else {
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c) {
              load_tile(dst + c * L::kChunkBytes, tmap, c, pi.bh, t0, &full[slot]);
              if (two) load_tile(dst + c * L::kChunkBytes + 8192, tmap, c, pi.bh, t1, &full[slot]);
            }
          }
          ++step;
        }
        if (!ok) break;
      }
      // Drain: every copy issued must land before the CTA can exit.
      const uint32_t first = step > kS ? step - kS : 0;
      for (uint32_t t = first; t < step; ++t) mbar_wait(&full[t % kS], (t / kS) & 1, kWaitNs);
      if (is_k && it > 0) mbar_wait(&sb.q_full, (it - 1) & 1, kWaitNs);
    }
  } else if (warp == kWarpMma) {
    // ===================================================== UMMA issuer
    const uint32_t idesc_s128 = kF8 ? idesc_e4m3(128, 128)
                                : kBF ? idesc_bf16(128, 128, 0, 0) : idesc_f16(128, 128, 0, 0);
    const uint32_t idesc_s64 = kF8 ? idesc_e4m3(128, 64)
                               : kBF ? idesc_bf16(128, 64, 0, 0) : idesc_f16(128, 64, 0, 0);
    const uint32_t idesc_pv = kF8 ? idesc_e4m3(128, D)
                              : kBF ? idesc_bf16(128, D, 0, 1) : idesc_f16(128, D, 0, 1);
    const uint64_t qd0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t kd0 = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vd0 = sdesc_sw128(smem_u32(sV), L::kChunkBytes, 1024);
    uint64_t qd[kKSteps];
#pragma unroll
    for (int k = 0; k < kKSteps; ++k) qd[k] = qd0 + (((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);

    // S = Q K^T of global step t into S buffer t % 2.  That buffer held P(t-2),
    // which PV(t-2), issued before this product, reads: the products run in
    // issue order.
    auto issue_s = [&](uint32_t t, bool two) -> bool {
      const uint32_t slot = t % kSK;
      if (!waitw(&sb.k_full[slot], (t / kSK) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      uint64_t kd[kKSteps];
      const uint64_t kb = kd0 + ((slot * L::kKVBytes) >> 4);
#pragma unroll
      for (int k = 0; k < kKSteps; ++k) kd[k] = kb + (((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);
      const uint32_t sd = tb + kColS + 128 * (t & 1);
      if constexpr (kF8)
        issue_ss4_f8(sd, qd, kd, two ? idesc_s128 : idesc_s64);
      else
        issue_ss_chain<kKSteps>(sd, qd, kd, two ? idesc_s128 : idesc_s64);
      commit_elect(&sb.s_full[t & 1]);
      commit_elect(&sb.k_empty[slot]);
      return true;
    };
    // O[obuf] += P V for global step t (P over the first columns of S buffer
    // t % 2, where the softmax warps write it after reading S(t)).
    auto issue_pv = [&](uint32_t t, bool two, bool first, int obuf) -> bool {
      const uint32_t slot = t % kSV, pbuf = t & 1;
      if (!waitw(&sb.p_full[pbuf], (t >> 1) & 1, abort_flag, P.status)) return false;
      if (!waitw(&sb.v_full[slot], (t / kSV) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      if constexpr (kF8) {
        // P (e4m3, 16 columns per key tile) x V^T: per key tile one 128-row box of
        // 64-byte rows, K steps of 32 keys at +32 bytes
        const uint64_t vb = sdesc_sw64(smem_u32(sV) + slot * L::kKVBytes, 512);
        const uint32_t pa = tb + kColS + pbuf * 128;
        issue_ts2_f8(tb + kColO + obuf * 128, pa, vb, vb + 2, idesc_pv, first ? 0u : 1u);
        if (two)
          issue_ts2_f8(tb + kColO + obuf * 128, pa + 16, vb + (8192 >> 4), vb + (8192 >> 4) + 2,
                       idesc_pv, 1u);
      } else {
        issue_ts_rows(tb + kColO + obuf * 128, tb + kColS + pbuf * 128,
                      vd0 + ((slot * L::kKVBytes) >> 4), two, idesc_pv, !first);
      }
      commit_elect(&sb.v_empty[slot]);  // also tells the rescale that PV(t) is done
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
      const int obuf = it & 1;
      // S of the item's first step, once Q has arrived
      if (!waitw(&sb.q_full, it & 1, abort_flag, P.status)) break;
      if (!issue_s(step, pi.count > 1)) break;
      if (nsteps == 1) commit_elect(&sb.q_empty);  // the item's last S product
      for (int s = 0; s < nsteps; ++s) {
        const uint32_t t = step + s;
        if (s + 1 < nsteps) {
          // S(t+1) into the other S buffer, ahead of PV(t)
          if (!issue_s(t + 1, 2 * s + 3 < pi.count)) {
            ok = false;
            break;
          }
          if (s + 2 == nsteps) commit_elect(&sb.q_empty);
        }
        if (s == 0 && it >= 2 &&
            !waitw(&sb.o_free[obuf], ((it >> 1) - 1) & 1, abort_flag, P.status)) {
          ok = false;  // the epilogue of item it-2 has not released O[obuf]
          break;
        }
        if (!issue_pv(t, 2 * s + 1 < pi.count, s == 0, obuf)) { ok = false; break; }
      }
      if (!ok) break;
      commit_elect(&sb.o_full[obuf]);
      step += nsteps;
      ++it;
    }
    // all issued MMAs complete before TMEM is released
    commit_elect(&sb.final_mma);
    mbar_wait(&sb.final_mma, 0, kWaitNs);
  } else if (warp < kSoftmaxWarps) {
    // ===================================================== softmax
    const int quarter = warp & 3;                // TMEM lane quarter of this warp
    const int hc = warp >> 2;                    // key tile of the step = column half
    const int row = quarter * 32 + lane;         // tile row 0..127
    const uint32_t mybit = (row >> 6) ? kSelB : kSelA;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = g.scale * 1.4426950408889634f;  // scale * log2(e)
    uint32_t step = 0, sq = 0;
    int it = 0;
    bool ok = true;
    // No abort test in the loop condition: both warps of a pair must walk the
    // same items and leave together (see pair_sync_or).
    while (ok) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (pair_sync_or(quarter, item == kSeqAbort) || item < 0) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;
      const uint32_t* list = P.lists + pi.off;
      const int nsteps = (pi.count + 1) / 2;
      const int obuf = it & 1;
      float m_run = -INFINITY, l_run = 0.f;
      // e4m3 variant: logits of the copies times the Q and K factors
      const float cs = kF8 ? c * __ldg(P.scales + 3 * pi.bh) * __ldg(P.scales + 3 * pi.bh + 1) : c;
      // list entry of this half's key tile, fetched one step ahead (its global
      // load latency would otherwise sit between two steps)
      uint32_t e_cur = hc < pi.count ? __ldg(list + hc) : 0u;
      for (int s = 0; s < nsteps; ++s, ++step) {
        const bool two = 2 * s + 1 < pi.count;
        const bool have = hc == 0 || two;  // this step has a key tile for this half
        const bool valid = have && (e_cur & mybit) != 0;
        e_cur = __ldg(list + min(2 * s + 2 + hc, pi.count - 1));  // in bounds; unused past the list
        const bool got = waitw(&sb.s_full[step & 1], (step >> 1) & 1, abort_flag, P.status);
        const uint32_t ts = tb + lane_addr + kColS + 128 * (step & 1);
        uint32_t x[64];  // this half-row of S; its first 32 words are reused for packed P
        float mx = -INFINITY;
        if (got) {
          tc_fence_after();
          if (valid) {
            tmem_ld32(ts + 64 * hc, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
            tmem_ld32(ts + 64 * hc + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
            tmem_wait_ld();
          }
        }
        if (got && valid) {
          float m8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            m8[i & 7] = max3f(m8[i & 7], __uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
          mx = fmaxf(max3f(m8[0], m8[1], m8[2]), max3f(max3f(m8[3], m8[4], m8[5]), m8[6], m8[7]));
        }
        sb.red[step & 1][hc][row] = mx;
        if (pair_sync_or(quarter, !got)) { ok = false; break; }
        const float m_new = fmaxf(m_run, fmaxf(mx, sb.red[step & 1][hc ^ 1][row]) * cs);
        bool resc = false;
        float alpha = 1.f;
        if (m_new > m_run + kRescaleThreshold) {
          if (m_run != -INFINITY) {
            alpha = ex2_approx(m_run - m_new);
            l_run *= alpha;
            resc = true;
          }
          m_run = m_new;
        }
        if (valid && kF8) {
          float ls[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) ls[u] = 0.f;
          const float mb = m_run;
          // x[i] <- e4m3x4(p[4i .. 4i+3]); x[4i .. 4i+3] are read before x[i] is
          // written
          unroll_for<16>([&](auto I) {
            constexpr int i = decltype(I)::value;
            float t0, t1, t2, t3;
            fma2_bc(t0, t1, __uint_as_float(x[4 * i]), __uint_as_float(x[4 * i + 1]), cs, -mb);
            fma2_bc(t2, t3, __uint_as_float(x[4 * i + 2]), __uint_as_float(x[4 * i + 3]), cs, -mb);
            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            const float p2 = ex2_approx(t2), p3 = ex2_approx(t3);
            add2_acc(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], p0, p1);
            add2_acc(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], p2, p3);
            x[i] = pack_e4m3x4(p0, p1, p2, p3);
          });
          l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        } else if (valid) {
          float ls[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) ls[u] = 0.f;
          const float mb = m_run;
          // x[i] <- f16x2(p[2i], p[2i+1]); x[2i], x[2i+1] are read before x[i] is
          // written.  Scale-and-shift and the row sum run on fp32 pairs.
          unroll_for<32>([&](auto I) {
            constexpr int i = decltype(I)::value;
            float t0, t1;
            fma2_bc(t0, t1, __uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]), c, -mb);
            const float p0 = ex2_approx(t0);
            const float p1 = ex2_approx(t1);
            add2_acc(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], p0, p1);
            x[i] = kBF ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
          });
          l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = 0u;
        }
        // P of key tile hc goes to columns [32 hc, 32 hc + 32) of S buffer
        // step % 2 (e4m3: [16 hc, 16 hc + 16)): both warps of the pair have
        // read their halves of S(t) before the exchange of maxima above
        if (have) {
          if constexpr (kF8)
            tmem_st16(ts + 16 * hc, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
          else
            tmem_st32(ts + 32 * hc, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        }
        if (__any_sync(0xffffffffu, resc)) {
          // O holds the previous steps' sum: wait for the last PV product,
          // then scale this half's columns of O in TMEM.  Both warps of the
          // pair see the same rows, so both take this branch.  (Done after P
          // is stored, so no part of x[] is live here.)
          // PV(step - 1) is done once its V slot is released (the slot's next
          // phase needs P of a later step, so the phase cannot move on first)
          const uint32_t pv = step - 1;
          const bool ready = waitw(&sb.v_empty[pv % kSV], (pv / kSV) & 1, abort_flag, P.status);
          if (pair_sync_or(quarter, !ready)) { ok = false; break; }
          tc_fence_after();
          const uint32_t to = tb + lane_addr + kColO + obuf * 128 + hc * (D / 2);
#pragma unroll 1
          for (int cc = 0; cc < D / 2; cc += 32) {
            uint32_t ov[32];
            tmem_ld32(to + cc, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(to + cc, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&sb.p_full[step & 1]);
      }
      if (!ok) break;
      // Hand this row's statistics to the epilogue through the stats buffer of
      // O[obuf]; the epilogue of item it-2 must have read it first.
      const bool got = it < 2 || waitw(&sb.st_free[obuf], ((it >> 1) - 1) & 1, abort_flag, P.status);
      if (pair_sync_or(quarter, !got)) break;
      sb.l_part[obuf][hc][row] = l_run;
      if (hc == 0) sb.m_fin[obuf][row] = m_run;
      warp_arrive(&sb.st_full[obuf]);
      ++it;
    }
  } else if (warp >= kWarpEpi && warp < kWarpEpi + kEpiWarps) {
    // ===================================================== epilogue
    // O_f leaves through a shared-memory stage as TMA stores (whole lines);
    // O (gated combine, caller layout) is written per row.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int half = row >> 6;                   // 0: first cube, 1: second cube
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const bool leader = threadIdx.x == kWarpEpi * 32;
    const bool stage_of = kOp == kOpF16 && P.o_f != nullptr;
    int it = 0;
    uint32_t sq = 0;
    // No abort test in the loop condition: the four warps meet at named
    // barriers and must walk the same items (see epi_sync_or).
    for (;;) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (epi_sync_or(item == kSeqAbort) || item < 0) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;
      const int obuf = it & 1;
      const bool live = half == 0 || pi.b >= 0;  // warp-uniform
      const int cube = (half && pi.b >= 0) ? pi.b : pi.a;
      const int o_in = row & 63;
      const size_t crow = static_cast<size_t>(pi.bh) * g.N + caller_row(g, cube, o_in);
      const size_t frow = static_cast<size_t>(pi.bh) * g.N + cube * kTile + o_in;
      const float* ocr = P.oc + (static_cast<size_t>(pi.bh) * g.Nc + cube) * D;
      // Gates and O_c of this row go to L2 while the item is still running, so
      // the chunk loads below hit L2.
      if (live) {
        const char* gcl = reinterpret_cast<const char*>(P.gc + crow * D);
        const char* gfl = reinterpret_cast<const char*>(P.gf + crow * D);
#pragma unroll
        for (int l = 0; l < D / 64; ++l) {
          prefetch_l2(gcl + 128 * l);
          prefetch_l2(gfl + 128 * l);
        }
      }
      if (lane < D / 32) prefetch_l2(ocr + 32 * lane);  // 4*D bytes of O_c: D/32 lines
      bool got = waitw(&sb.st_full[obuf], (it >> 1) & 1, abort_flag, P.status);
      float l_sum = 1.f, m_fin = 0.f;
      if (got) {
        l_sum = sb.l_part[obuf][0][row] + sb.l_part[obuf][1][row];
        m_fin = sb.m_fin[obuf][row];
        warp_arrive(&sb.st_free[obuf]);
        got = waitw(&sb.o_full[obuf], (it >> 1) & 1, abort_flag, P.status);
      }
      if (epi_sync_or(!got)) break;
      tc_fence_after();
      // e4m3 variant: the V copy's factor joins the normalisation
      const float inv_l = (kF8 ? __ldg(P.scales + 3 * pi.bh + 2) : 1.f) / l_sum;
      const uint32_t to = tb + lane_addr + kColO + obuf * 128;
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t ov[32];
        if (live) {
          tmem_ld32(to + cc, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * inv_l);
        }
        if (stage_of) {
          // O_f in fp16: a staged row of 128 bytes holds 64 columns, the chunks
          // cc and cc + 32 of a pair; the pair leaves as one box per cube
          const bool first = (cc & 63) == 0;
          if (first) {
            // the previous pair's stores have read the stage
            if (leader) bulk_wait_group_read0();
            epi_sync();
          }
          if (live) {
            uint8_t* rp = sStage + row * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int unit = ((cc & 63) >> 3) + u;
              const uint4 w = make_uint4(
                  pack_f16x2(__uint_as_float(ov[8 * u]), __uint_as_float(ov[8 * u + 1])),
                  pack_f16x2(__uint_as_float(ov[8 * u + 2]), __uint_as_float(ov[8 * u + 3])),
                  pack_f16x2(__uint_as_float(ov[8 * u + 4]), __uint_as_float(ov[8 * u + 5])),
                  pack_f16x2(__uint_as_float(ov[8 * u + 6]), __uint_as_float(ov[8 * u + 7])));
              *reinterpret_cast<uint4*>(rp + ((unit ^ (row & 7)) << 4)) = w;
            }
          }
          if (!first) {
            fence_proxy_async_smem();
            epi_sync();
            if (leader) {
              tma_store_2d(&tof, sStage, cc - 32, pi.bh * g.N + pi.a * kTile);
              if (pi.b >= 0) tma_store_2d(&tof, sStage + 64 * 128, cc - 32, pi.bh * g.N + pi.b * kTile);
              bulk_commit_group();
            }
          }
        }
        if (live) {
          uint4* op = reinterpret_cast<uint4*>(P.o + crow * D + cc);
          const uint4* gcp = reinterpret_cast<const uint4*>(P.gc + crow * D + cc);
          const uint4* gfp = reinterpret_cast<const uint4*>(P.gf + crow * D + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 gcr = gcp[v], gfr = gfp[v];
            const __nv_bfloat162* g2c = reinterpret_cast<const __nv_bfloat162*>(&gcr);
            const __nv_bfloat162* g2f = reinterpret_cast<const __nv_bfloat162*>(&gfr);
            uint4 res;
            uint32_t* rp = reinterpret_cast<uint32_t*>(&res);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int d = cc + 8 * v + 2 * e;
              const float2 fc = __bfloat1622float2(g2c[e]);
              const float2 ff = __bfloat1622float2(g2f[e]);
              const float2 oc2 = *reinterpret_cast<const float2*>(ocr + d);
              const float y0 = fmaf(oc2.x, fc.x, __uint_as_float(ov[8 * v + 2 * e]) * ff.x);
              const float y1 = fmaf(oc2.y, fc.y, __uint_as_float(ov[8 * v + 2 * e + 1]) * ff.y);
              rp[e] = pack_bf16x2(y0, y1);
            }
            op[v] = res;
          }
        }
      }
      if (live && P.lse_f) P.lse_f[frow] = (m_fin + __log2f(l_sum)) * 0.6931471805599453f;
      tc_fence_before();
      warp_arrive(&sb.o_free[obuf]);
      ++it;
    }
    if (leader) bulk_wait_group0();  // O_f stores complete before the CTA exits
  } else if (warp == kWarpSeq) {
    // ===================================================== item fetcher
    if (lane == 0) seq_fetch(sb.seq, P.sched, P.n_items, abort_flag, P.status);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tb, kTmemCols);
}

template <int D>
cudaError_t run_fwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                    FwdParams p, cudaStream_t s) {
  alignas(64) CUtensorMap mq, mk, mv, mof;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  if (!encode_tiled_2d(&mq, q, rows, D, 64, 64) || !encode_tiled_2d(&mk, k, rows, D, 64, 64) ||
      !encode_tiled_2d(&mv, v, rows, D, 64, 64))
    return cudaErrorInvalidValue;
  // O_f (fp16, cube order): boxes of 64 rows (one cube) x 64 columns
  memset(&mof, 0, sizeof(mof));
  if (p.o_f && !encode_tiled_2d(&mof, p.o_f, rows, D, 64, 64)) return cudaErrorInvalidValue;
  const int smem = FwdSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(fine_fwd_kernel<D, kOpF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(p.n_items);
  if (grid <= 0) return cudaSuccess;
  if ((e = cudaMemsetAsync(p.sched, 0, sizeof(int), s)) != cudaSuccess) return e;
  fine_fwd_kernel<D, kOpF16><<<grid, kThreadsFwd, smem, s>>>(mq, mk, mv, mof, p);
  return cudaGetLastError();
}

// bf16 variant: the caller's q, k, v in place (5-D cube boxes of the raster
// layout, or 2-D 64-row boxes of the cube layout).
template <int D>
cudaError_t run_fwd_bf16(const Geom& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                         const __nv_bfloat16* v, FwdParams p, cudaStream_t s) {
  alignas(64) CUtensorMap mq, mk, mv, mof;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  const bool ok = g.raster ? (encode_raster_cubes_bf16(&mq, q, g) &&
                              encode_raster_cubes_bf16(&mk, k, g) &&
                              encode_raster_cubes_bf16(&mv, v, g))
                           : (encode_tiled_2d_bf16(&mq, q, rows, D) &&
                              encode_tiled_2d_bf16(&mk, k, rows, D) &&
                              encode_tiled_2d_bf16(&mv, v, rows, D));
  if (!ok) return cudaErrorInvalidValue;
  memset(&mof, 0, sizeof(mof));
  const int smem = FwdSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(fine_fwd_kernel<D, kOpBF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(p.n_items);
  if (grid <= 0) return cudaSuccess;
  if ((e = cudaMemsetAsync(p.sched, 0, sizeof(int), s)) != cudaSuccess) return e;
  fine_fwd_kernel<D, kOpBF16><<<grid, kThreadsFwd, smem, s>>>(mq, mk, mv, mof, p);
  return cudaGetLastError();
}

// e4m3 variant, head_dim 128: Q8, K8 [BH*N, 128] bytes (boxes of 64 rows x 128
// bytes, 128-byte swizzle); V8T [BH*Nc*128, 64] bytes (boxes of 128 rows x 64
// bytes, 64-byte swizzle).
cudaError_t run_fwd_fp8(const Geom& g, const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                        FwdParams p, cudaStream_t s) {
  constexpr int D = 128;
  alignas(64) CUtensorMap mq, mk, mv, mof;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  const uint64_t vrows = static_cast<uint64_t>(g.BH) * g.Nc * D;
  if (!encode_tiled_2d_u8(&mq, q8, rows, D, 64, D, 128) ||
      !encode_tiled_2d_u8(&mk, k8, rows, D, 64, D, 128) ||
      !encode_tiled_2d_u8(&mv, v8t, vrows, kTile, D, kTile, 64))
    return cudaErrorInvalidValue;
  memset(&mof, 0, sizeof(mof));
  const int smem = FwdSmem<D, true>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(fine_fwd_kernel<D, kOpE4M3>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(p.n_items);
  if (grid <= 0) return cudaSuccess;
  if ((e = cudaMemsetAsync(p.sched, 0, sizeof(int), s)) != cudaSuccess) return e;
  fine_fwd_kernel<D, kOpE4M3><<<grid, kThreadsFwd, smem, s>>>(mq, mk, mv, mof, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fine_fwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                            const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                            __nv_bfloat16* o, __half* o_f, float* lse_f, const Workspace& ws,
                            cudaStream_t s) {
  FwdParams p{g, ws.qpairs, ws.qlist, ws.n_qpairs, use_cost_order(g) ? ws.qorder : nullptr,
              gc, gf, oc, o, o_f, lse_f, ws.status, nullptr, ws.counter + kCounterFwd};
  if (g.D == 64) return launch_fine_fwd64(g, q, k, v, gc, gf, oc, o, o_f, lse_f, ws, s);
  return run_fwd<128>(g, q, k, v, p, s);
}

cudaError_t launch_fine_fwd_bf16(const Geom& g, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                 const __nv_bfloat16* v, const __nv_bfloat16* gc,
                                 const __nv_bfloat16* gf, const float* oc, __nv_bfloat16* o,
                                 float* lse_f, const Workspace& ws, cudaStream_t s) {
  FwdParams p{g, ws.qpairs, ws.qlist, ws.n_qpairs, use_cost_order(g) ? ws.qorder : nullptr,
              gc, gf, oc, o, nullptr, lse_f, ws.status, nullptr, ws.counter + kCounterFwd};
  if (g.D == 64) return launch_fine_fwd64_bf16(g, q, k, v, gc, gf, oc, o, lse_f, ws, s);
  return run_fwd_bf16<128>(g, q, k, v, p, s);
}

cudaError_t launch_fine_fwd_fp8(const Geom& g, const uint8_t* q8, const uint8_t* k8,
                                const uint8_t* v8t, const float* scales,
                                const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                                __nv_bfloat16* o, float* lse_f, const Workspace& ws,
                                cudaStream_t s) {
  if (g.D != 128) return cudaErrorInvalidValue;
  FwdParams p{g, ws.qpairs, ws.qlist, ws.n_qpairs, use_cost_order(g) ? ws.qorder : nullptr,
              gc, gf, oc, o, nullptr, lse_f, ws.status, scales, ws.counter + kCounterFwd};
  return run_fwd_fp8(g, q8, k8, v8t, p, s);
}

}  // namespace vsa

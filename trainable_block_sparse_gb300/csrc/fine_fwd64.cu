// Fine stage of VSA, forward, head_dim 64, fused with the gated combine ("VSA:
// Faster Video Diffusion with Trainable Sparse Attention", §2 "Fine stage" and
// App. B: token-level attention only inside the selected 64x64 blocks; paper
// notes 关键设计 3: O = O_c (.) G_c + O_f (.) G_f).  Same work items, lists and
// outputs as the fine forward of fine_fwd.cu.
//
// Why a kernel of its own: at head_dim 64 a step's products are short, and in
// a CTA that runs one chain of steps the hand-offs between its UMMA warp and
// its softmax warps (S done -> softmax -> P stored -> next products) take
// three to four times as long as the products themselves.  Here every per-CTA
// resource is halved (256 TMEM columns, 97 KB of shared memory, 384 threads)
// so that two CTAs share each SM, and within a CTA the S product runs two
// steps ahead of the softmax:
//  * a step is one key cube (64 keys); S has two TMEM buffers, so S(t+2) is
//    issued as soon as S(t) has been read, and the softmax warps find S(t+1)
//    ready when they finish step t;
//  * the item's Q is copied into TMEM once per item (an A operand), so both
//    products of a step read only their K or V tile from shared memory
//    (S = Q K^T: four M128 N64 K16 products, O += P V: four M128 N64 K16);
//  * a thread owns a whole row of the step (64 keys, in registers), so the
//    row maximum needs no exchange between warps.
//
// Per CTA, twelve warps:
//   warps 0-3  softmax: warp w owns TMEM lane quarter w (32 token rows); it
//              also copies its rows of the item's Q into TMEM;
//   warps 4-7  epilogue: normalise O_f, gated combine with the cube's coarse
//              output, O (bf16, caller layout), O_f (fp16, cube order, kept
//              for the backward), log-sum-exp;
//   warp 8     TMA: Q once per item, then K tiles; warp 9: V tiles;
//   warp 10    UMMA issue; warp 11: item fetcher (the next item from the
//              launch's shared counter, item_seq.cuh).
// TMEM: S buffers at columns 0 and 64, Q at 160 (32 columns of fp16 pairs), O at
// 192 (64).  P(t) (32 columns of fp16 pairs) is written over the first half of
// S(t)'s buffer as soon as it is computed, with a full barrier per buffer; the
// next product into that buffer, S(t+2), is issued once PV(t) has completed,
// and O is rescaled only after PV(t-1) is done.  One O accumulator: an item's
// first P V product waits until the epilogue has read the previous item's O.
// The running maximum moves, and O is rescaled, only when a row's maximum grows
// by more than 2^8 (the rule of fine_fwd.cu, applied per 64-key step).
// Every mbarrier wait is bounded; a time-out is recorded in the status word and
// the CTA unwinds, waits for its own copies and products, frees TMEM and exits.
//
// bf16 variant (inference: no O_f): Q, K, V read in place from the caller's bf16
// tensors (5-D cube boxes of the raster layout, or 64-row boxes of the cube
// layout), P in bf16, kind::f16 UMMAs with bf16 operands.
#include <cfloat>
#include <cstring>

#include "item_seq.cuh"
#include "umma_pipe.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kD = 64;
constexpr int kThreads64 = 384;  // 12 warps
constexpr int kWarpEpi64 = 4, kWarpK64 = 8, kWarpV64 = 9, kWarpMma64 = 10;  // 11: item fetcher
// readers of the item sequence: K and V producer threads, UMMA warp, 4
// softmax and 4 epilogue warps
constexpr int kSeqReaders64 = 11;
constexpr uint32_t kCols64 = 256;
constexpr uint32_t kColS64 = 0;    // two S buffers of 64 columns
constexpr uint32_t kColQ64 = 160;  // Q: 64 channels as 32 columns of fp16 pairs
constexpr uint32_t kColO64 = 192;  // O: 64 fp32 columns
constexpr float kRescale64 = 8.0f;  // log2 units
// Register split per warpgroup; the launch gives 65536 / (2 x 384) -> 80 a
// thread, 30720 per CTA, and the three shares must fit in that.
constexpr int kRegsSoftmax64 = 128, kRegsEpi64 = 80, kRegsRest64 = 32;
constexpr int kLaunchRegs64 = 80;
static_assert(128 * (kRegsSoftmax64 + kRegsEpi64 + kRegsRest64) <= kThreads64 * kLaunchRegs64,
              "register split exceeds the launch's registers");
// setmaxnreg.inc may only raise a warp's count and .dec only lower it: the
// shares that decrease must not exceed the launch's count (a .dec above it is
// an illegal instruction), the one that increases must not be below it.
static_assert(kRegsSoftmax64 >= kLaunchRegs64 && kRegsEpi64 <= kLaunchRegs64 &&
                  kRegsRest64 <= kLaunchRegs64 && kRegsEpi64 % 8 == 0 && kRegsRest64 % 8 == 0 &&
                  kRegsSoftmax64 % 8 == 0 && kRegsRest64 >= 24,
              "setmaxnreg shares must move away from the launch's count, in steps of 8");
enum : int { kOp64F16 = 0, kOp64BF16 = 2 };

constexpr int kStagesK64 = 4, kStagesV64 = 4;
struct L64 {
  static constexpr int kTileBytes = 64 * kD * 2;  // one 64-row tile (8 KB)
  static constexpr int kQ = 0;                    // Q: two tiles (128 rows)
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kStagesK64 * kTileBytes;
  static constexpr int kStage = kV + kStagesV64 * kTileBytes;  // O_f: 128 rows x 128 bytes
  static constexpr int kBytes = kStage + 2 * kTileBytes + 1024;
};

struct Bars64 {
  uint64_t q_full, q_empty;  // Q in shared memory / copied out of it
  uint64_t q_tmem, q_done;   // Q in TMEM / the item's last S product done
  uint64_t k_full[kStagesK64], k_empty[kStagesK64], v_full[kStagesV64], v_empty[kStagesV64];
  uint64_t s_full[2];  // per S buffer
  uint64_t p_full[2];  // P(t) stored over S buffer t % 2 (one arrival per softmax warp)
  uint64_t o_full, o_free;        // the item's O complete / read by the epilogue
  uint64_t st_full, st_free;      // row statistics handed to / read by the epilogue
  uint64_t final_mma;
  ItemSeq seq;
  uint32_t tmem_base;
  int abort;
  float l_fin[128], m_fin[128];
};

struct FwdParams64 {
  Geom g;
  const PairItem* items;
  const uint32_t* lists;
  int n_items;
  const int* order;  // schedule position -> item (null: identity)
  const __nv_bfloat16* gc;
  const __nv_bfloat16* gf;
  const float* oc;
  __nv_bfloat16* o;
  __half* o_f;
  float* lse_f;
  uint32_t* status;
  int* sched;  // schedule counter, zero at launch
};

__device__ __forceinline__ void warp_arrive64(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Named barrier over the four epilogue warps returning the OR of `fail`, so
// they leave the item loop together.
__device__ __forceinline__ bool epi_sync_or64(bool fail) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 5, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(fail))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void epi_sync64() { asm volatile("bar.sync 5, 128;" ::: "memory"); }

template <int kOp>
__global__ void __launch_bounds__(kThreads64, 2)
    fine_fwd64_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tof,
                      FwdParams64 P) {
  constexpr bool kBF = kOp == kOp64BF16;
  constexpr int kSK = kStagesK64, kSV = kStagesV64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L64::kQ;
  uint8_t* sK = smem + L64::kK;
  uint8_t* sV = smem + L64::kV;
  uint8_t* sStage = smem + L64::kStage;
  __shared__ Bars64 sb;
  int* abort_flag = &sb.abort;
  const Geom& g = P.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&sb.q_full, 1);
    mbar_init(&sb.q_empty, 4);  // one arrival per softmax warp
    mbar_init(&sb.q_tmem, 4);
    mbar_init(&sb.q_done, 1);
    for (int i = 0; i < kSK; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
    }
    for (int i = 0; i < kSV; ++i) {
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 4);
    }
    mbar_init(&sb.o_full, 1);
    mbar_init(&sb.o_free, 4);  // one arrival per epilogue warp
    mbar_init(&sb.st_full, 4);
    mbar_init(&sb.st_free, 4);
    mbar_init(&sb.final_mma, 1);
    seq_init(sb.seq, kSeqReaders64);
    sb.abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma64) {
    tmem_alloc(&sb.tmem_base, kCols64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = sb.tmem_base;

  // Each role sets its warpgroup's register share first (warps 0-3 up, the
  // rest down), inside its own branch.
  if (warp == kWarpK64 || warp == kWarpV64) {
    // ===================================================== TMA producers
    regs_dec<kRegsRest64>();
    const bool is_k = warp == kWarpK64;
    if (lane == 0) {
      const CUtensorMap* tmap = is_k ? &tk : &tv;
      uint64_t* full = is_k ? sb.k_full : sb.v_full;
      uint64_t* empty = is_k ? sb.k_empty : sb.v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const uint32_t kS = is_k ? kSK : kSV;
      tma_prefetch_desc(tmap);
      if (is_k) tma_prefetch_desc(&tq);
      // one 64-row tile of a cube of slice bh: a 2-D box of a cube-order tensor,
      // or (bf16 variant, raster layout) a 5-D box of the caller's tensor
      auto load_tile = [&](uint8_t* dst, const CUtensorMap* m, int bh, int cube, uint64_t* bar) {
        if (kBF && g.raster) {
          const int cw_ = cube % g.cw, rest = cube / g.cw;
          tma_load_5d(dst, m, 0, 4 * cw_, 4 * (rest % g.ch), 4 * (rest / g.ch), bh, bar);
        } else {
          tma_load_2d(dst, m, 0, bh * g.N + cube * kTile, bar);
        }
      };
      uint32_t step = 0, sq = 0;
      int it = 0;
      for (;;) {
        const int item = seq_next<false>(sb.seq, sq, abort_flag, P.status);
        if (item < 0 || is_aborted(abort_flag)) break;
        const PairItem pi = P.items[P.order ? P.order[item] : item];
        if (pi.count == 0) continue;
        const uint32_t* list = P.lists + pi.off;
        if (is_k) {
          if (it > 0 && !wait1(&sb.q_empty, (it - 1) & 1, abort_flag, P.status)) break;
          mbar_arrive_expect_tx(&sb.q_full, 2 * L64::kTileBytes);
          load_tile(sQ, &tq, pi.bh, pi.a, &sb.q_full);
          load_tile(sQ + L64::kTileBytes, &tq, pi.bh, pi.b >= 0 ? pi.b : pi.a, &sb.q_full);
        }
        ++it;
        bool ok = true;
        for (int s = 0; s < pi.count; ++s) {
          const uint32_t slot = step % kS, ph = (step / kS) & 1;
          if (step >= kS && !wait1(&empty[slot], ph ^ 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[slot], L64::kTileBytes);
          load_tile(ring + slot * L64::kTileBytes, tmap, pi.bh,
                    static_cast<int>(list[s] & 0xFFFFu), &full[slot]);
          ++step;
        }
        if (!ok) break;
      }
      // every copy issued lands before the CTA exits
      const uint32_t first = step > kS ? step - kS : 0;
      for (uint32_t t = first; t < step; ++t) mbar_wait(&full[t % kS], (t / kS) & 1, kWaitNs);
      if (is_k && it > 0) mbar_wait(&sb.q_full, (it - 1) & 1, kWaitNs);
    }
  } else if (warp == kWarpMma64) {
    // ===================================================== UMMA issuer
    regs_dec<kRegsRest64>();
    const uint32_t id_s = kBF ? idesc_bf16(128, 64, 0, 0) : idesc_f16(128, 64, 0, 0);
    const uint32_t id_pv = kBF ? idesc_bf16(128, kD, 0, 1) : idesc_f16(128, kD, 0, 1);
    const uint64_t kd0 = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vd0 = sdesc_sw128(smem_u32(sV), L64::kTileBytes, 1024);

    // S(t) = Q K^T into S buffer t % 2 (A = Q in TMEM, B = K tile, K-major),
    // once PV(t-2) has read P(t-2) out of that buffer (PV(t-2) was issued
    // earlier, after the softmax warps had read S(t-2) and stored P(t-2))
    auto issue_s = [&](uint32_t t) -> bool {
      const uint32_t slot = t % kSK, buf = t & 1;
      if (t >= 2) {
        const uint32_t pv = t - 2;
        if (!waitw(&sb.v_empty[pv % kSV], (pv / kSV) & 1, abort_flag, P.status)) return false;
      }
      if (!waitw(&sb.k_full[slot], (t / kSK) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      const uint64_t kb = kd0 + ((slot * L64::kTileBytes) >> 4);
      issue_ts4(tb + kColS64 + 64 * buf, tb + kColQ64, kb, kb + 2, kb + 4, kb + 6, id_s, 0u);
      commit_elect(&sb.s_full[buf]);
      commit_elect(&sb.k_empty[slot]);
      return true;
    };
    // O += P V of step t (A = P(t), packed over the first 32 columns of S
    // buffer t % 2; B = V tile, MN-major); its commit releases the V slot and
    // that S buffer, and tells the softmax warps that O may be rescaled
    auto issue_pv = [&](uint32_t t, bool first) -> bool {
      const uint32_t slot = t % kSV;
      if (!waitw(&sb.v_full[slot], (t / kSV) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      const uint64_t vb = vd0 + ((slot * L64::kTileBytes) >> 4);
      issue_ts4(tb + kColO64, tb + kColS64 + 64 * (t & 1), vb, vb + (2048 >> 4),
                vb + (4096 >> 4), vb + (6144 >> 4), id_pv, first ? 0u : 1u);
      commit_elect(&sb.v_empty[slot]);
      return true;
    };

    uint32_t step = 0, sq = 0;
    int it = 0;
    bool ok = true;
    while (ok) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (item < 0 || is_aborted(abort_flag)) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;
      const int n = pi.count;
      if (!waitw(&sb.q_tmem, it & 1, abort_flag, P.status)) break;
      // S of the item's first two steps
      if (!issue_s(step) || (n > 1 && !issue_s(step + 1))) break;
      if (n <= 2) commit_elect(&sb.q_done);  // the item's last S product
      for (int s = 0; s < n; ++s) {
        const uint32_t t = step + s;
        if (!waitw(&sb.p_full[t & 1], (t >> 1) & 1, abort_flag, P.status)) {
          ok = false;
          break;
        }
        if (s == 0 && it >= 1 && !waitw(&sb.o_free, (it - 1) & 1, abort_flag, P.status)) {
          ok = false;  // the epilogue has not read the previous item's O
          break;
        }
        if (!issue_pv(t, s == 0)) {
          ok = false;
          break;
        }
        if (s + 2 < n) {
          if (!issue_s(t + 2)) {
            ok = false;
            break;
          }
          if (s + 3 == n) commit_elect(&sb.q_done);
        }
      }
      if (!ok) break;
      commit_elect(&sb.o_full);
      step += n;
      ++it;
    }
    // all issued products complete before TMEM is released
    commit_elect(&sb.final_mma);
    mbar_wait(&sb.final_mma, 0, kWaitNs);
  } else if (warp < 4) {
    // ===================================================== softmax
    regs_inc<kRegsSoftmax64>();
    const int quarter = warp;
    const int row = quarter * 32 + lane;
    const uint32_t mybit = (row >> 6) ? kSelB : kSelA;  // the same for the whole warp
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t to = tb + lane_addr + kColO64;
    const float c = g.scale * 1.4426950408889634f;  // scale * log2(e)
    uint32_t step = 0, sq = 0;
    int it = 0;
    bool ok = true;
    while (ok) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (item < 0 || is_aborted(abort_flag)) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;
      const uint32_t* list = P.lists + pi.off;
      // This row of the item's Q into TMEM (the A operand of S), once the
      // previous item's last S product is done with it.
      if (it > 0 && !waitw(&sb.q_done, (it - 1) & 1, abort_flag, P.status)) break;
      if (!waitw(&sb.q_full, it & 1, abort_flag, P.status)) break;
      {
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4*>(sQ + row * 128 + ((u ^ (row & 7)) << 4));
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
        tc_fence_after();
        tmem_st32(tb + lane_addr + kColQ64, w);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive64(&sb.q_tmem);
        warp_arrive64(&sb.q_empty);
      }
      float m_run = -INFINITY, l_run = 0.f;
      uint32_t e_next = __ldg(list);  // list entry of the step, fetched one step ahead
      for (int s = 0; s < pi.count; ++s, ++step) {
        const bool valid = (e_next & mybit) != 0;
        e_next = __ldg(list + min(s + 1, pi.count - 1));
        const uint32_t buf = step & 1;
        if (!waitw(&sb.s_full[buf], (step >> 1) & 1, abort_flag, P.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t x[64];  // the row's 64 logits; the first 32 words are reused for P
        if (valid) {
          const uint32_t ts = tb + lane_addr + kColS64 + 64 * buf;
          tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
          tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
          tmem_wait_ld();
        }
        float alpha = 1.f;
        bool resc = false;
        if (valid) {
          float m8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) m8[u] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            m8[i & 7] = max3f(m8[i & 7], __uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
          const float mx =
              fmaxf(max3f(m8[0], m8[1], m8[2]), max3f(max3f(m8[3], m8[4], m8[5]), m8[6], m8[7]));
          const float m_new = fmaxf(m_run, mx * c);
          if (m_new > m_run + kRescale64) {
            if (m_run != -INFINITY) {
              alpha = ex2_approx(m_run - m_new);
              l_run *= alpha;
              resc = true;
            }
            m_run = m_new;
          }
          float ls[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) ls[u] = 0.f;
          const float mb = m_run;
          // x[i] <- pair(p[2i], p[2i+1]); x[2i], x[2i+1] are read before x[i] is written
          unroll_for<32>([&](auto I) {
            constexpr int i = decltype(I)::value;
            float t0, t1;
            fma2_bc(t0, t1, __uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]), c, -mb);
            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
            add2_acc(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], p0, p1);
            x[i] = kBF ? pack_bf16x2(p0, p1) : pack_f16x2(p0, p1);
          });
          l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = 0u;
        }
        // P(t) goes over the first half of S(t)'s columns (this warp's rows,
        // read above); nothing else touches them until PV(t) has completed.
        // O is rescaled only once PV(t-1) is done.
        tmem_st32(tb + lane_addr + kColS64 + 64 * buf, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        const bool resc_any = __any_sync(0xffffffffu, resc);
        if (resc_any && step > 0) {
          const uint32_t pv = step - 1;
          if (!waitw(&sb.v_empty[pv % kSV], (pv / kSV) & 1, abort_flag, P.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (resc_any) {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            uint32_t ov[32];
            tmem_ld32(to + 32 * h, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(to + 32 * h, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive64(&sb.p_full[buf]);
      }
      if (!ok) break;
      // the row's statistics to the epilogue (which has read the previous ones)
      if (it > 0 && !waitw(&sb.st_free, (it - 1) & 1, abort_flag, P.status)) break;
      sb.l_fin[row] = l_run;
      sb.m_fin[row] = m_run;
      warp_arrive64(&sb.st_full);
      ++it;
    }
  } else if (warp < 8) {
    // ===================================================== epilogue
    regs_dec<kRegsEpi64>();
    const int quarter = warp - kWarpEpi64;
    const int row = quarter * 32 + lane;
    const int half = row >> 6;  // 0: first cube of the item, 1: second
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t to = tb + lane_addr + kColO64;
    const bool leader = threadIdx.x == kWarpEpi64 * 32;
    const bool stage_of = !kBF && P.o_f != nullptr;
    int it = 0;
    uint32_t sq = 0;
    // No abort test in the loop condition: the four warps meet at named
    // barriers and walk the same items.
    for (;;) {
      const int item = seq_next<true>(sb.seq, sq, abort_flag, P.status);
      if (epi_sync_or64(item == kSeqAbort) || item < 0) break;
      const PairItem pi = P.items[P.order ? P.order[item] : item];
      if (pi.count == 0) continue;
      const bool live = half == 0 || pi.b >= 0;  // warp-uniform
      const int cube = (half && pi.b >= 0) ? pi.b : pi.a;
      const int o_in = row & 63;
      const size_t crow = static_cast<size_t>(pi.bh) * g.N + caller_row(g, cube, o_in);
      const size_t frow = static_cast<size_t>(pi.bh) * g.N + cube * kTile + o_in;
      const float* ocr = P.oc + (static_cast<size_t>(pi.bh) * g.Nc + cube) * kD;
      if (live) {
        prefetch_l2(P.gc + crow * kD);
        prefetch_l2(P.gf + crow * kD);
      }
      if (lane < 2) prefetch_l2(ocr + 32 * lane);
      bool got = waitw(&sb.st_full, it & 1, abort_flag, P.status);
      float l_sum = 1.f, m_fin = 0.f;
      if (got) {
        l_sum = sb.l_fin[row];
        m_fin = sb.m_fin[row];
        warp_arrive64(&sb.st_free);
        got = waitw(&sb.o_full, it & 1, abort_flag, P.status);
      }
      if (epi_sync_or64(!got)) break;
      tc_fence_after();
      const float inv_l = 1.f / l_sum;
      if (stage_of) {
        // the previous item's O_f stores have read the stage
        if (leader) bulk_wait_group_read0();
        epi_sync64();
      }
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t ov[32];
        if (live) {
          tmem_ld32(to + 32 * h, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * inv_l);
        }
        if (h == 1) {
          // O is in registers: the next item may accumulate into it
          tc_fence_before();
          warp_arrive64(&sb.o_free);
        }
        if (stage_of && live) {
          // O_f (fp16): 128-byte staged rows, 16-byte units swizzled by row % 8
          uint8_t* rp = sStage + row * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int unit = 4 * h + u;
            const uint4 w = make_uint4(
                pack_f16x2(__uint_as_float(ov[8 * u]), __uint_as_float(ov[8 * u + 1])),
                pack_f16x2(__uint_as_float(ov[8 * u + 2]), __uint_as_float(ov[8 * u + 3])),
                pack_f16x2(__uint_as_float(ov[8 * u + 4]), __uint_as_float(ov[8 * u + 5])),
                pack_f16x2(__uint_as_float(ov[8 * u + 6]), __uint_as_float(ov[8 * u + 7])));
            *reinterpret_cast<uint4*>(rp + ((unit ^ (row & 7)) << 4)) = w;
          }
        }
        if (live) {
          const int cc = 32 * h;
          uint4* op = reinterpret_cast<uint4*>(P.o + crow * kD + cc);
          const uint4* gcp = reinterpret_cast<const uint4*>(P.gc + crow * kD + cc);
          const uint4* gfp = reinterpret_cast<const uint4*>(P.gf + crow * kD + cc);
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
      if (stage_of) {
        fence_proxy_async_smem();
        epi_sync64();
        if (leader) {
          tma_store_2d(&tof, sStage, 0, pi.bh * g.N + pi.a * kTile);
          if (pi.b >= 0) tma_store_2d(&tof, sStage + 64 * 128, 0, pi.bh * g.N + pi.b * kTile);
          bulk_commit_group();
        }
      }
      if (live && P.lse_f) P.lse_f[frow] = (m_fin + __log2f(l_sum)) * 0.6931471805599453f;
      ++it;
    }
    if (leader) bulk_wait_group0();  // O_f stores complete before the CTA exits
  } else {
    // ===================================================== item fetcher
    // (warp 11; its register share completes warpgroup 2's split)
    regs_dec<kRegsRest64>();
    if (lane == 0) seq_fetch(sb.seq, P.sched, P.n_items, abort_flag, P.status);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma64) tmem_dealloc(tb, kCols64);
}

// Checks that the compiled kernel was given the registers its split assumes
// (setmaxnreg.inc would otherwise wait for registers that never come), sets
// its shared memory, and launches two CTAs per SM.
template <int kOp>
cudaError_t launch64(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const CUtensorMap& mof, const FwdParams64& p, cudaStream_t s) {
  auto kern = fine_fwd64_kernel<kOp>;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  // every share must move away from the launch's count in its own direction,
  // and the shares must fit in the launch's registers
  if (attr.numRegs < kRegsEpi64 || attr.numRegs < kRegsRest64 || attr.numRegs > kRegsSoftmax64 ||
      attr.numRegs * kThreads64 < 128 * (kRegsSoftmax64 + kRegsEpi64 + kRegsRest64))
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L64::kBytes);
  if (e != cudaSuccess) return e;
  // two CTAs' shared memory (~2 x 100 KB) needs the largest shared-memory carveout
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (p.n_items <= 0) return cudaSuccess;
  const int sms = persistent_grid(1 << 30);  // min(n, SMs) of a huge n: the SM count
  const int grid = p.n_items < 2 * sms ? p.n_items : 2 * sms;
  if ((e = cudaMemsetAsync(p.sched, 0, sizeof(int), s)) != cudaSuccess) return e;
  kern<<<grid, kThreads64, L64::kBytes, s>>>(mq, mk, mv, mof, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fine_fwd64(const Geom& g, const __half* q, const __half* k, const __half* v,
                              const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                              __nv_bfloat16* o, __half* o_f, float* lse_f, const Workspace& ws,
                              cudaStream_t s) {
  if (g.D != kD) return cudaErrorInvalidValue;
  FwdParams64 p{g, ws.qpairs, ws.qlist, ws.n_qpairs, use_cost_order(g) ? ws.qorder : nullptr,
                gc, gf, oc, o, o_f, lse_f, ws.status, ws.counter + kCounterFwd};
  alignas(64) CUtensorMap mq, mk, mv, mof;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  if (!encode_tiled_2d(&mq, q, rows, kD, 64, 64) || !encode_tiled_2d(&mk, k, rows, kD, 64, 64) ||
      !encode_tiled_2d(&mv, v, rows, kD, 64, 64))
    return cudaErrorInvalidValue;
  memset(&mof, 0, sizeof(mof));
  if (o_f && !encode_tiled_2d(&mof, o_f, rows, kD, 64, 64)) return cudaErrorInvalidValue;
  return launch64<kOp64F16>(mq, mk, mv, mof, p, s);
}

cudaError_t launch_fine_fwd64_bf16(const Geom& g, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v,
                                   const __nv_bfloat16* gc, const __nv_bfloat16* gf,
                                   const float* oc, __nv_bfloat16* o, float* lse_f,
                                   const Workspace& ws, cudaStream_t s) {
  if (g.D != kD) return cudaErrorInvalidValue;
  FwdParams64 p{g, ws.qpairs, ws.qlist, ws.n_qpairs, use_cost_order(g) ? ws.qorder : nullptr,
                gc, gf, oc, o, nullptr, lse_f, ws.status, ws.counter + kCounterFwd};
  alignas(64) CUtensorMap mq, mk, mv, mof;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  const bool ok = g.raster ? (encode_raster_cubes_bf16(&mq, q, g) &&
                              encode_raster_cubes_bf16(&mk, k, g) &&
                              encode_raster_cubes_bf16(&mv, v, g))
                           : (encode_tiled_2d_bf16(&mq, q, rows, kD) &&
                              encode_tiled_2d_bf16(&mk, k, rows, kD) &&
                              encode_tiled_2d_bf16(&mv, v, rows, kD));
  if (!ok) return cudaErrorInvalidValue;
  memset(&mof, 0, sizeof(mof));
  return launch64<kOp64BF16>(mq, mk, mv, mof, p, s);
}

}  // namespace vsa

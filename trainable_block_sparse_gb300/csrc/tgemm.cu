// fp32-accurate batched GEMM on the tensor cores, for the coarse stage of VSA
// ("VSA: Faster Video Diffusion with Trainable Sparse Attention", §2 "Coarse
// stage": attention among the mean-pooled cubes, its softmax and, for
// training, its gradients).  The coarse logits decide which blocks the fine
// stage attends to, so they need fp32 accuracy: a single tf32 or bf16 product
// would move them by ~1e-3.  Each fp32 operand x is split into two tf32 values
// x = hi + lo (hi = round(x), lo = round(x - hi), |x - hi - lo| <= 2^-22 |x|)
// and a.b is accumulated as lo_a.hi_b + hi_a.lo_b + hi_a.hi_b; the dropped
// lo_a.lo_b term is below 2^-22 |a b|, comparable to fp32 rounding.
// Operands given without a lo part (null) run as plain tf32 instead: one
// product per k-step from the hi parts (round-to-nearest tf32, relative error
// 2^-11 per element), for products whose results need no more (the coarse
// backward: its gradients reach the outputs divided by 64).
//
// D[b] = A[b] B[b]^T (A [M x K], B [N x K], both K-major), 128 x 128 output
// tiles, k-blocks of 32 (one 128-byte swizzled row per operand row).  The
// dual form also computes E[b] = A2[b] B2[b]^T of the same tile into a second
// accumulator, for epilogues that combine the two (the coarse attention
// backward: P from the logits and dL = P (.) (dP - delta) from dP; dL is
// written as it stands and, like P, transposed, so the products that
// contract over query cubes read K-major operands).
// Persistent, one CTA per SM, six or ten warps:
//   warp 0    TMA: the operand tiles of each k-block (A hi, A lo, B hi, B lo,
//             or A hi, B hi; zero-filled outside the matrices) into a ring of
//             three stages (pairs) or four (hi parts);
//   warp 1    UMMA: 12 (pairs) or 4 kind::tf32 products per k-block into
//             one of two TMEM accumulators (the epilogue of tile i overlaps
//             tile i+1);
//   warps 2-  epilogue (four warps for pairs, eight for hi parts, two per
//             TMEM lane quarter splitting the columns): one accumulator row
//             per thread; each 32 x 32 block of an output is written into a
//             128-byte-swizzled shared-memory tile (directly or transposed;
//             a ring of three per warp for hi parts) and leaves as one TMA
//             store (rows and columns outside the matrix are clipped by the
//             tensor map).
// Every mbarrier wait is bounded; a time-out sets the status word and the CTA
// unwinds as the fine kernels do.
#include <cstring>

#include "umma_pipe.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kTM = 128, kTN = 128, kTK = 32;
constexpr int kOpBytes = kTM * kTK * 4;            // one 128 x 32 fp32 operand tile
constexpr int kBlockBytes = 32 * 32 * 4;           // one 32 x 32 fp32 output block

// Shared memory and epilogue warps per operand form.  tf32 pairs take four
// operand tiles a k-block (A hi, A lo, B hi, B lo: 64 KB) in three stages,
// which leaves room for four epilogue warps with one output staging block
// each; their products (three per k-step) outlast the epilogue.  Hi parts
// alone take two tiles (A hi, B hi: 32 KB) and one product per k-step, so
// the epilogue (exponentials and up to two outputs per element in the
// attention-backward forms) would bind with one warp per lane quarter:
// eight warps, two per quarter splitting the tile's columns, each with three
// staging blocks (it fills one while the TMA stores of the others still read
// them), beside four stages.
template <bool kPair>
struct TgPlan {
  static constexpr int kStages = kPair ? 3 : 4;
  static constexpr int kStageBytes = (kPair ? 4 : 2) * kOpBytes;
  static constexpr int kBOff = (kPair ? 2 : 1) * kOpBytes;  // B hi within a stage
  static constexpr int kEpiWarps = kPair ? 4 : 8;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;   // TMA, UMMA, epilogue warps
  static constexpr int kEpiBlocks = kPair ? 1 : 3;
  static constexpr int kEpiBytes = kEpiBlocks * kBlockBytes;  // per epilogue warp
  static constexpr int kSmem = kStages * kStageBytes + kEpiWarps * kEpiBytes + 1024;
  static_assert(kEpiWarps % 4 == 0 && (kTN / 32) % (kEpiWarps / 4) == 0, "column split");
  static_assert(kSmem <= 227 * 1024, "tgemm shared memory");
  static_assert(kEpiBytes % 1024 == 0, "staging blocks stay 1024-byte aligned");
};
constexpr int kTgMaxStages = 4;

// The sources of all but the N most recently committed bulk stores have been read.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

struct TgBars {
  uint64_t full[kTgMaxStages], empty[kTgMaxStages];
  uint64_t acc_full[2], acc_free[2];
  uint64_t final_mma;
  uint32_t tmem_base;
  int abort;
};

// 12 products of one k-block: 4 k-steps of K = 8 (32 bytes of each swizzled
// row), each lo_a.hi_b + hi_a.lo_b + hi_a.hi_b; one elected lane issues all.
__device__ __forceinline__ void issue_kblock_tf32(uint32_t d, uint64_t ah, uint64_t al,
                                                  uint64_t bh, uint64_t bl, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b64 ah, al, bh, bl;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %6, 0;\n\tsetp.eq.b32 t, %6, %6;\n\t"
      "mov.b64 ah, %1;\n\tmov.b64 al, %2;\n\tmov.b64 bh, %3;\n\tmov.b64 bl, %4;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], al, bh, %5, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bl, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %5, t;\n\t"
      "add.s64 ah, ah, 2;\n\tadd.s64 al, al, 2;\n\tadd.s64 bh, bh, 2;\n\tadd.s64 bl, bl, 2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], al, bh, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bl, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %5, t;\n\t"
      "add.s64 ah, ah, 2;\n\tadd.s64 al, al, 2;\n\tadd.s64 bh, bh, 2;\n\tadd.s64 bl, bl, 2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], al, bh, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bl, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %5, t;\n\t"
      "add.s64 ah, ah, 2;\n\tadd.s64 al, al, 2;\n\tadd.s64 bh, bh, 2;\n\tadd.s64 bl, bl, 2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], al, bh, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bl, %5, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %5, t;\n\t}" ::"r"(d),
      "l"(ah), "l"(al), "l"(bh), "l"(bl), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Plain tf32: 4 products of one k-block from the hi parts only.
__device__ __forceinline__ void issue_kblock_tf32_hi(uint32_t d, uint64_t ah, uint64_t bh,
                                                     uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\t.reg .b64 ah, bh;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %4, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
      "mov.b64 ah, %1;\n\tmov.b64 bh, %2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %3, f;\n\t"
      "add.s64 ah, ah, 2;\n\tadd.s64 bh, bh, 2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %3, t;\n\t"
      "add.s64 ah, ah, 2;\n\tadd.s64 bh, bh, 2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %3, t;\n\t"
      "add.s64 ah, ah, 2;\n\tadd.s64 bh, bh, 2;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::tf32 [%0], ah, bh, %3, t;\n\t}" ::"r"(d),
      "l"(ah), "l"(bh), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct TileCoord {
  int b, tm, tn;
};

__device__ __forceinline__ TileCoord tile_of(int t, int tiles_m, int tiles_n) {
  TileCoord c;
  c.tn = t % tiles_n;
  c.tm = (t / tiles_n) % tiles_m;
  c.b = t / (tiles_n * tiles_m);
  return c;
}

struct TgMaps {
  CUtensorMap ah, al, bh, bl;
};

// Output tensor maps (fp32 [batch][M][ld], box 32 x 32); unused ones stay zero.
struct TgOutMaps {
  CUtensorMap out, hi, lo, vt, pt;
};

// kPair: operands as tf32 pairs (three products per k-step); otherwise the
// hi parts alone (one product), whose stage holds A hi and B hi at the same
// offsets.
template <bool kDual, bool kPair>
__global__ void __launch_bounds__(TgPlan<kPair>::kThreads, 1)
    tgemm_kernel(const __grid_constant__ TgMaps m0, const __grid_constant__ TgMaps m1,
                 const __grid_constant__ TgOutMaps om, TgemmArgs P, uint32_t* status) {
  using Plan = TgPlan<kPair>;
  constexpr int kTgStages = Plan::kStages;
  constexpr int kStageBytes = Plan::kStageBytes;
  constexpr int kEpiBlocks = Plan::kEpiBlocks;
  constexpr int kProducts = kDual ? 2 : 1;
  constexpr uint32_t kLoadBytes = kStageBytes;
  constexpr uint32_t kAccCols = kTN * kProducts;     // per tile buffer
  constexpr uint32_t kTmemCols = 2 * kAccCols;       // two tile buffers
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* epi_smem = reinterpret_cast<float*>(smem + kTgStages * kStageBytes);
  __shared__ TgBars sb;
  int* abort_flag = &sb.abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tiles_m = (P.M + kTM - 1) / kTM, tiles_n = (P.N + kTN - 1) / kTN;
  const int ntiles = P.batch * tiles_m * tiles_n;
  const int kblocks = (P.K + kTK - 1) / kTK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTgStages; ++i) {
      mbar_init(&sb.full[i], 1);
      mbar_init(&sb.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.acc_full[i], 1);
      mbar_init(&sb.acc_free[i], Plan::kEpiWarps);
    }
    mbar_init(&sb.final_mma, 1);
    sb.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sb.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = sb.tmem_base;

  if (warp == 0) {
    // ===================================================== TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&m0.ah);
      tma_prefetch_desc(&m0.bh);
      if (kPair) {
        tma_prefetch_desc(&m0.al);
        tma_prefetch_desc(&m0.bl);
      }
      uint32_t n = 0;  // k-blocks issued
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok && !is_aborted(abort_flag); t += gridDim.x) {
        const TileCoord c = tile_of(t, tiles_m, tiles_n);
        for (int pr = 0; pr < kProducts && ok; ++pr) {
          const TgMaps& m = pr ? m1 : m0;
          for (int kb = 0; kb < kblocks; ++kb, ++n) {
            const uint32_t slot = n % kTgStages;
            if (n >= static_cast<uint32_t>(kTgStages) &&
                !wait1(&sb.empty[slot], ((n / kTgStages) & 1) ^ 1, abort_flag, status)) {
              ok = false;
              break;
            }
            uint8_t* st = smem + slot * kStageBytes;
            mbar_arrive_expect_tx(&sb.full[slot], kLoadBytes);
            tma_load_3d(st, &m.ah, kb * kTK, c.tm * kTM, c.b, &sb.full[slot]);
            tma_load_3d(st + Plan::kBOff, &m.bh, kb * kTK, c.tn * kTN, c.b, &sb.full[slot]);
            if (kPair) {
              tma_load_3d(st + kOpBytes, &m.al, kb * kTK, c.tm * kTM, c.b, &sb.full[slot]);
              tma_load_3d(st + 3 * kOpBytes, &m.bl, kb * kTK, c.tn * kTN, c.b, &sb.full[slot]);
            }
          }
        }
      }
      const uint32_t first = n > static_cast<uint32_t>(kTgStages) ? n - kTgStages : 0;
      for (uint32_t i = first; i < n; ++i)
        mbar_wait(&sb.full[i % kTgStages], (i / kTgStages) & 1, kWaitNs);
    }
  } else if (warp == 1) {
    // ===================================================== UMMA issuer
    const uint32_t idesc = idesc_tf32(kTM, kTN);
    const uint64_t d0 = sdesc_sw128(smem_u32(smem), 16, 1024);
    uint32_t n = 0;
    int lt = 0;  // tiles of this CTA
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok && !is_aborted(abort_flag); t += gridDim.x, ++lt) {
      const int buf = lt & 1;
      if (lt >= 2 && !waitw(&sb.acc_free[buf], ((lt >> 1) - 1) & 1, abort_flag, status)) break;
      tc_fence_after();
      for (int pr = 0; pr < kProducts && ok; ++pr) {
        const uint32_t dt = tb + buf * kAccCols + pr * kTN;
        for (int kb = 0; kb < kblocks; ++kb, ++n) {
          const uint32_t slot = n % kTgStages;
          if (!waitw(&sb.full[slot], (n / kTgStages) & 1, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t base = d0 + ((slot * kStageBytes) >> 4);
          if (kPair)
            issue_kblock_tf32(dt, base, base + (kOpBytes >> 4), base + ((2 * kOpBytes) >> 4),
                              base + ((3 * kOpBytes) >> 4), idesc, kb > 0 ? 1u : 0u);
          else
            issue_kblock_tf32_hi(dt, base, base + (Plan::kBOff >> 4), idesc, kb > 0 ? 1u : 0u);
          commit_elect(&sb.empty[slot]);
        }
      }
      if (!ok) break;
      commit_elect(&sb.acc_full[buf]);
    }
    commit_elect(&sb.final_mma);
    mbar_wait(&sb.final_mma, 0, kWaitNs);
  } else {
    // ===================================================== epilogue
    // warp w reads TMEM lane quarter w % 4; with eight warps, warps 2-5 take
    // the first half of each tile's column chunks and warps 6-9 the second
    const int quarter = warp & 3, ew = warp - 2;
    constexpr int kChunks = (kTN / 32) / (Plan::kEpiWarps / 4);
    const int ch0 = (ew / 4) * kChunks;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    // this warp's staging blocks (1024-aligned)
    uint8_t* blk0 = reinterpret_cast<uint8_t*>(epi_smem) + ew * Plan::kEpiBytes;
    uint32_t nblk = 0;  // output blocks this warp has staged
    int lt = 0;
    for (int t = blockIdx.x; t < ntiles && !is_aborted(abort_flag); t += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const TileCoord c = tile_of(t, tiles_m, tiles_n);
      const int mbase = c.tm * kTM + quarter * 32;
      const int m = mbase + lane;
      float r1 = 0.f, r2 = 0.f;
      if (P.mode == kTgAttnBwd && m < P.M) {
        r1 = P.v1[c.b * P.vec_stride + m];
        r2 = P.v2[c.b * P.vec_stride + m];
      }
      if (!waitw(&sb.acc_full[buf], (lt >> 1) & 1, abort_flag, status)) break;
      tc_fence_after();
#pragma unroll 1
      for (int ch = ch0; ch < ch0 + kChunks; ++ch) {
        const int n0 = c.tn * kTN + 32 * ch;
        if (n0 >= P.N) break;
        uint32_t v[32], e[32];
        tmem_ld32(tb + lane_addr + buf * kAccCols + 32 * ch, v);
        if (kDual) tmem_ld32(tb + lane_addr + buf * kAccCols + kTN + 32 * ch, e);
        tmem_wait_ld();
        float val[32], pv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float a = __uint_as_float(v[j]);
          if (!kDual || P.mode == kTgScale) {
            val[j] = P.alpha * a;
          } else {
            pv[j] = ex2_approx(fmaf(P.alpha, a, -P.beta * r1));
            val[j] = pv[j] * (__uint_as_float(e[j]) - r2);
          }
        }
        // one output block: rows mbase.., columns n0.. through the staging block
        auto store_block = [&](const CUtensorMap* map, const float (&src)[32], int part) {
          // the store that last used this block has read it
          if (lane == 0) bulk_wait_group_read<kEpiBlocks - 1>();
          __syncwarp();
          uint8_t* blk = blk0 + (nblk++ % kEpiBlocks) * kBlockBytes;
          uint8_t* rp = blk + lane * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float q[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x = src[4 * u + e];
              const float h = round_tf32(x);
              q[e] = part == 0 ? x : (part == 1 ? h : round_tf32(x - h));
            }
            *reinterpret_cast<float4*>(rp + ((u ^ (lane & 7)) << 4)) =
                make_float4(q[0], q[1], q[2], q[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(map, blk, n0, mbase, c.b);
            bulk_commit_group();
          }
        };
        // the transposed block (columns n0.. as rows, rows mbase.. as
        // columns): thread `lane` writes column `lane` of it, one word per
        // row, the 32 lanes of a row covering all 32 banks
        auto store_block_t = [&](const CUtensorMap* map, const float (&src)[32]) {
          if (lane == 0) bulk_wait_group_read<kEpiBlocks - 1>();
          __syncwarp();
          uint8_t* blk = blk0 + (nblk++ % kEpiBlocks) * kBlockBytes;
#pragma unroll
          for (int r = 0; r < 32; ++r)
            *reinterpret_cast<float*>(blk + r * 128 + ((((lane >> 2) ^ (r & 7))) << 4) +
                                      (lane & 3) * 4) = round_tf32(src[r]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(map, blk, mbase, n0, c.b);
            bulk_commit_group();
          }
        };
        if (P.out) store_block(&om.out, val, 0);
        if (P.out_hi) store_block(&om.hi, val, 1);
        if (P.out_lo) store_block(&om.lo, val, 2);
        if (kDual && P.vt_hi) store_block_t(&om.vt, val);
        if (kDual && P.pt_hi) store_block_t(&om.pt, pv);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.acc_free[buf]);
    }
  }

  if (warp >= 2 && lane == 0) bulk_wait_group0();  // output stores complete before exit
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tb, kTmemCols);
}

// One tf32-pair split per job: fp32 [batch][rows][cols] -> hi, lo in the same
// orientation or transposed, through padded 32 x 32 shared-memory tiles.  A
// block takes kSplitTiles tiles side by side along the columns (32 rows x 128
// columns) and issues all their loads before any store, so each thread keeps
// sixteen loads in flight instead of four.
struct SplitJob {
  const float* src;
  float* hi;
  float* lo;
  long long stride_src, stride_dst;
  int ld_src, ld_dst, rows, cols, transpose;
};
constexpr int kMaxSplitJobs = 8;
constexpr int kSplitTiles = 4;
struct SplitJobs {
  SplitJob j[kMaxSplitJobs];
};

__global__ void __launch_bounds__(256) split_kernel(const __grid_constant__ SplitJobs jobs,
                                                    int batch) {
  __shared__ float t[kSplitTiles][32][33];
  const SplitJob& J = jobs.j[blockIdx.z / batch];
  const int b = blockIdx.z % batch, r0 = blockIdx.y * 32;
  const int cb = blockIdx.x * 32 * kSplitTiles;
  if (r0 >= J.rows || cb >= J.cols) return;  // this job is smaller than the grid
  const float* s = J.src + b * J.stride_src;
#pragma unroll
  for (int q = 0; q < kSplitTiles; ++q) {
#pragma unroll
    for (int r = threadIdx.y; r < 32; r += 8) {
      const int rr = r0 + r, cc = cb + 32 * q + threadIdx.x;
      t[q][r][threadIdx.x] =
          (rr < J.rows && cc < J.cols) ? s[static_cast<size_t>(rr) * J.ld_src + cc] : 0.f;
    }
  }
  __syncthreads();
  float* h = J.hi + b * J.stride_dst;
  float* l = J.lo ? J.lo + b * J.stride_dst : nullptr;  // null: hi parts only
#pragma unroll
  for (int q = 0; q < kSplitTiles; ++q) {
    const int c0 = cb + 32 * q;
#pragma unroll
    for (int r = threadIdx.y; r < 32; r += 8) {
      if (!J.transpose) {
        const int rr = r0 + r, cc = c0 + threadIdx.x;
        if (rr < J.rows && cc < J.cols) {
          const float x = t[q][r][threadIdx.x];
          const float xh = round_tf32(x);
          h[static_cast<size_t>(rr) * J.ld_dst + cc] = xh;
          if (l) l[static_cast<size_t>(rr) * J.ld_dst + cc] = round_tf32(x - xh);
        }
      } else {
        const int cc = c0 + r, rr = r0 + threadIdx.x;  // output row = input column
        if (rr < J.rows && cc < J.cols) {
          const float x = t[q][threadIdx.x][r];
          const float xh = round_tf32(x);
          h[static_cast<size_t>(cc) * J.ld_dst + rr] = xh;
          if (l) l[static_cast<size_t>(cc) * J.ld_dst + rr] = round_tf32(x - xh);
        }
      }
    }
  }
}

}  // namespace

namespace {

// Operand maps; with `pair` false only the hi parts are read (the lo maps stay zero).
bool encode_maps(TgMaps* m, const TgemmArgs& a, const TgemmOperand& A, const TgemmOperand& B,
                 bool pair) {
  memset(m, 0, sizeof(*m));
  if ((A.ld & 3) || (B.ld & 3) || (A.stride & 3) || (B.stride & 3)) return false;
  if (!A.hi || !B.hi || (pair && (!A.lo || !B.lo))) return false;
  return encode_tiled_3d_f32(&m->ah, A.hi, a.batch, a.M, a.K, A.ld, A.stride, kTK, kTM) &&
         encode_tiled_3d_f32(&m->bh, B.hi, a.batch, a.N, a.K, B.ld, B.stride, kTK, kTN) &&
         (!pair ||
          (encode_tiled_3d_f32(&m->al, A.lo, a.batch, a.M, a.K, A.ld, A.stride, kTK, kTM) &&
           encode_tiled_3d_f32(&m->bl, B.lo, a.batch, a.N, a.K, B.ld, B.stride, kTK, kTN)));
}

bool encode_outs(TgOutMaps* o, const TgemmArgs& a) {
  memset(o, 0, sizeof(*o));
  // [batch][rows][ld] with rows x cols valid: M x N, or N x M for the transposes
  auto enc = [&](CUtensorMap* m, float* p, int ld, long long stride, bool t) {
    if (!p) return true;
    if ((ld & 3) || (stride & 3)) return false;
    return encode_tiled_3d_f32(m, p, a.batch, t ? a.N : a.M, t ? a.M : a.N, ld, stride, 32,
                               32);
  };
  return enc(&o->out, a.out, a.out_ld, a.out_stride, false) &&
         enc(&o->hi, a.out_hi, a.split_ld, a.split_stride, false) &&
         enc(&o->lo, a.out_lo, a.split_ld, a.split_stride, false) &&
         enc(&o->vt, a.vt_hi, a.t_ld, a.t_stride, true) &&
         enc(&o->pt, a.pt_hi, a.t_ld, a.t_stride, true);
}

template <bool kDual, bool kPair>
cudaError_t run_tgemm(const TgemmArgs& a, const TgMaps& m0, const TgMaps& m1, uint32_t* status,
                      cudaStream_t s) {
  alignas(64) TgOutMaps om;
  if (!encode_outs(&om, a)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tgemm_kernel<kDual, kPair>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TgPlan<kPair>::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long ntiles = static_cast<long long>(a.batch) * ((a.M + kTM - 1) / kTM) *
                           ((a.N + kTN - 1) / kTN);
  const int grid = static_cast<int>(ntiles < sms ? ntiles : sms);
  tgemm_kernel<kDual, kPair><<<grid, TgPlan<kPair>::kThreads, TgPlan<kPair>::kSmem, s>>>(
      m0, m1, om, a, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tgemm(const TgemmArgs& a, const TgemmOperand& A, const TgemmOperand& B,
                         uint32_t* status, cudaStream_t s) {
  if (a.batch <= 0 || a.M <= 0 || a.N <= 0 || a.K <= 0) return cudaSuccess;
  if (a.mode != kTgScale) return cudaErrorInvalidValue;
  const bool pair = A.lo != nullptr;
  alignas(64) TgMaps m0;
  if (!encode_maps(&m0, a, A, B, pair)) return cudaErrorInvalidValue;
  return pair ? run_tgemm<false, true>(a, m0, m0, status, s)
              : run_tgemm<false, false>(a, m0, m0, status, s);
}

cudaError_t launch_tgemm_dual(const TgemmArgs& a, const TgemmOperand& A, const TgemmOperand& B,
                              const TgemmOperand& A2, const TgemmOperand& B2, uint32_t* status,
                              cudaStream_t s) {
  if (a.batch <= 0 || a.M <= 0 || a.N <= 0 || a.K <= 0) return cudaSuccess;
  if (a.mode != kTgAttnBwd) return cudaErrorInvalidValue;
  const bool pair = A.lo != nullptr;
  alignas(64) TgMaps m0, m1;
  if (!encode_maps(&m0, a, A, B, pair) || !encode_maps(&m1, a, A2, B2, pair))
    return cudaErrorInvalidValue;
  return pair ? run_tgemm<true, true>(a, m0, m1, status, s)
              : run_tgemm<true, false>(a, m0, m1, status, s);
}

cudaError_t launch_split_tf32(const SplitSpec* specs, int n, int batch, cudaStream_t s) {
  if (n <= 0 || batch <= 0) return cudaSuccess;
  if (n > kMaxSplitJobs || batch > 65535) return cudaErrorInvalidValue;
  if (static_cast<long long>(batch) * n > 65535) {  // grid.z limit: one launch per job
    for (int i = 0; i < n; ++i) {
      const cudaError_t e = launch_split_tf32(specs + i, 1, batch, s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  SplitJobs jobs{};
  int max_r = 0, max_c = 0;
  for (int i = 0; i < n; ++i) {
    const SplitSpec& p = specs[i];
    jobs.j[i] = SplitJob{p.src, p.hi, p.lo, p.stride_src, p.stride_dst, p.ld_src, p.ld_dst,
                         p.rows, p.cols, p.transpose ? 1 : 0};
    max_r = p.rows > max_r ? p.rows : max_r;
    max_c = p.cols > max_c ? p.cols : max_c;
  }
  if (max_r <= 0 || max_c <= 0) return cudaSuccess;
  const int strip = 32 * kSplitTiles;
  const dim3 grid((max_c + strip - 1) / strip, (max_r + 31) / 32, batch * n);
  split_kernel<<<grid, dim3(32, 8), 0, s>>>(jobs, batch);
  return cudaGetLastError();
}

}  // namespace vsa

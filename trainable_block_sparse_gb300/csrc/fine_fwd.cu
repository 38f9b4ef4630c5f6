// Fine stage of VSA, forward, fused with the gated combine ("VSA: Faster Video
// Diffusion with Trainable Sparse Attention", §2 "Fine stage" and App. B:
// token-level attention only inside the selected 64x64 blocks; paper notes
// 关键设计 3: O = O_c (.) G_c + O_f (.) G_f).
//
// GB300 design (tcgen05 + TMEM + TMA, one persistent CTA per SM):
//  * Work item = two query cubes of one (batch, head): their 2 x 64 token rows
//    form one M = 128 tensor-core tile, and the item walks the union of the two
//    index lists (list entries carry which cube selected the key cube; rows of
//    the other cube treat that block as masked).
//  * Steps take two key cubes at a time, so S = Q K^T is an M=128, N=128 UMMA
//    chain and O += P V an M=128, N=D, K=128 chain (N=64 UMMAs run at ~60% of
//    the tensor pipe, N=128 at ~97%).
//  * Warp 0 issues TMA tile loads (Q once per item; K and V tiles gathered by
//    list entry into a ring of stages), warp 1 issues UMMAs, warps 2-5 run the
//    online softmax one token row per thread straight out of TMEM and write P
//    back into TMEM as the A operand of the PV product.
//  * Q, K, V arrive as fp16 cube-order staged copies and P is written in fp16:
//    with the running maximum kept stale (below), the largest P entries are
//    rounded too, and fp16's 11-bit significand keeps that error 8x below
//    bf16's.  Every UMMA is fp16 x fp16 with fp32 accumulation.
//  * S is double-buffered in TMEM so QK^T of step t+1 overlaps the softmax of
//    step t.  The running maximum is only moved (and O rescaled in TMEM) when
//    it grows by more than 2^8, which keeps exp arguments bounded and makes the
//    rescale rare.
//  * The epilogue normalises O_f, applies the gates with the cube's coarse
//    output, and writes O (bf16, caller layout: un-permuted on the way out),
//    O_f (fp32, kept for the backward) and the log-sum-exp.
// Every mbarrier wait is bounded; a time-out is recorded in the status word and
// the CTA unwinds, waits for its own in-flight copies and MMAs, frees TMEM and
// exits.
#include <cfloat>

#include "umma_pipe.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr int kThreadsFwd = 192;           // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;              // S buffers at columns 0 and 128
constexpr uint32_t kColO = 256;            // O accumulator
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdSmem {
  static constexpr int kChunks = D / 64;              // 64-column (128-byte) chunks
  static constexpr int kChunkBytes = 128 * 128;       // one chunk of 128 rows
  static constexpr int kQBytes = kChunks * kChunkBytes;
  static constexpr int kKVBytes = kChunks * kChunkBytes;  // 2 key tiles
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kTileBytes = 64 * D * 2;       // one 64-row tile
  static constexpr int kBytes = kQBytes + 2 * kStages * kKVBytes + 1024;
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t o_ready, o_full, final_mma;
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  Geom g;
  const PairItem* items;
  const uint32_t* lists;
  int n_items;
  const __nv_bfloat16* gc;
  const __nv_bfloat16* gf;
  const float* oc;
  __nv_bfloat16* o;
  float* o_f;
  float* lse_f;
  uint32_t* status;
};

template <int D>
__global__ void __launch_bounds__(kThreadsFwd, 1)
    fine_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, FwdParams P) {
  using L = FwdSmem<D>;
  constexpr int kS = L::kStages;
  constexpr int kKSteps = D / 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + L::kQBytes;
  uint8_t* sV = sK + kS * L::kKVBytes;
  __shared__ FwdBars sb;
  int* abort_flag = &sb.abort;

  const Geom& g = P.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&sb.q_full, 1);
    mbar_init(&sb.q_empty, 1);
    for (int i = 0; i < kS; ++i) {
      mbar_init(&sb.k_full[i], 1);
      mbar_init(&sb.k_empty[i], 1);
      mbar_init(&sb.v_full[i], 1);
      mbar_init(&sb.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 128);
    }
    mbar_init(&sb.o_ready, 1);
    mbar_init(&sb.o_full, 1);
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
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      uint32_t step = 0;
      int it = 0;  // items with work seen by this CTA
      for (int item = blockIdx.x; item < P.n_items && !is_aborted(abort_flag);
           item += gridDim.x) {
        const PairItem pi = P.items[item];
        if (pi.count == 0) continue;
        const uint32_t* list = P.lists + pi.off;
        if (it > 0 && !wait1(&sb.q_empty, (it - 1) & 1, abort_flag, P.status)) break;
        mbar_arrive_expect_tx(&sb.q_full, L::kQBytes);
        const int row_a = pi.bh * g.N + pi.a * kTile;
        const int row_b = pi.bh * g.N + (pi.b >= 0 ? pi.b : pi.a) * kTile;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_2d(sQ + c * L::kChunkBytes, &tq, c * 64, row_a, &sb.q_full);
          tma_load_2d(sQ + c * L::kChunkBytes + 8192, &tq, c * 64, row_b, &sb.q_full);
        }
        ++it;
        const int nsteps = (pi.count + 1) / 2;
        bool ok = true;
        for (int s = 0; s < nsteps; ++s) {
          const uint32_t slot = step % kS, ph = (step / kS) & 1;
          const bool two = 2 * s + 1 < pi.count;
          const int t0 = static_cast<int>(list[2 * s] & 0xFFFFu);
          const int t1 = two ? static_cast<int>(list[2 * s + 1] & 0xFFFFu) : t0;
          const uint32_t bytes = (two ? 2 : 1) * L::kTileBytes;
          if (step >= static_cast<uint32_t>(kS) &&
              (!wait1(&sb.k_empty[slot], ph ^ 1, abort_flag, P.status) ||
               !wait1(&sb.v_empty[slot], ph ^ 1, abort_flag, P.status))) {
            ok = false;
            break;
          }
          uint8_t* dk = sK + slot * L::kKVBytes;
          uint8_t* dv = sV + slot * L::kKVBytes;
          const int r0 = pi.bh * g.N + t0 * kTile, r1 = pi.bh * g.N + t1 * kTile;
          mbar_arrive_expect_tx(&sb.k_full[slot], bytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_2d(dk + c * L::kChunkBytes, &tk, c * 64, r0, &sb.k_full[slot]);
            if (two) tma_load_2d(dk + c * L::kChunkBytes + 8192, &tk, c * 64, r1, &sb.k_full[slot]);
          }
          mbar_arrive_expect_tx(&sb.v_full[slot], bytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            tma_load_2d(dv + c * L::kChunkBytes, &tv, c * 64, r0, &sb.v_full[slot]);
            if (two) tma_load_2d(dv + c * L::kChunkBytes + 8192, &tv, c * 64, r1, &sb.v_full[slot]);
          }
          ++step;
        }
        if (!ok) break;
      }
      // Drain: every copy issued must land before the CTA can exit.
      const uint32_t first = step > static_cast<uint32_t>(kS) ? step - kS : 0;
      for (uint32_t t = first; t < step; ++t) {
        mbar_wait(&sb.k_full[t % kS], (t / kS) & 1, kWaitNs);
        mbar_wait(&sb.v_full[t % kS], (t / kS) & 1, kWaitNs);
      }
      if (it > 0) mbar_wait(&sb.q_full, (it - 1) & 1, kWaitNs);
    }
  } else if (warp == 1) {
    // ===================================================== UMMA issuer
    const uint32_t idesc_s128 = idesc_f16(128, 128, 0, 0);
    const uint32_t idesc_s64 = idesc_f16(128, 64, 0, 0);
    const uint32_t idesc_pv = idesc_f16(128, D, 0, 1);
    const uint64_t qd0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t kd0 = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t vd0 = sdesc_sw128(smem_u32(sV), L::kChunkBytes, 1024);
    uint64_t qd[kKSteps];
#pragma unroll
    for (int k = 0; k < kKSteps; ++k) qd[k] = qd0 + (((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);

    // O += P V for global step gstep (P from the S buffer of that step).
    auto issue_pv = [&](uint32_t gstep, bool two, bool first) -> bool {
      const uint32_t slot = gstep % kS, sbuf = gstep & 1;
      if (!waitw(&sb.p_full[sbuf], (gstep >> 1) & 1, abort_flag, P.status)) return false;
      if (!waitw(&sb.v_full[slot], (gstep / kS) & 1, abort_flag, P.status)) return false;
      tc_fence_after();
      issue_ts_rows(tb + kColO, tb + kColS + sbuf * 128, vd0 + ((slot * L::kKVBytes) >> 4), two,
                    idesc_pv, !first);
      commit_elect(&sb.v_empty[slot]);
      commit_elect(&sb.o_ready);
      return true;
    };

    uint32_t step = 0;
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < P.n_items && ok && !is_aborted(abort_flag);
         item += gridDim.x) {
      const PairItem pi = P.items[item];
      if (pi.count == 0) continue;
      const int nsteps = (pi.count + 1) / 2;
      if (!waitw(&sb.q_full, it & 1, abort_flag, P.status)) break;
      ++it;
      tc_fence_after();
      bool prev_two = false;
      for (int s = 0; s < nsteps; ++s, ++step) {
        const uint32_t slot = step % kS, sbuf = step & 1;
        const bool two = 2 * s + 1 < pi.count;
        if (!waitw(&sb.k_full[slot], (step / kS) & 1, abort_flag, P.status)) { ok = false; break; }
        tc_fence_after();
        uint64_t kd[kKSteps];
        const uint64_t kb = kd0 + ((slot * L::kKVBytes) >> 4);
#pragma unroll
        for (int k = 0; k < kKSteps; ++k) kd[k] = kb + (((k / 4) * L::kChunkBytes + (k % 4) * 32) >> 4);
        issue_ss_chain<kKSteps>(tb + kColS + sbuf * 128, qd, kd, two ? idesc_s128 : idesc_s64);
        commit_elect(&sb.s_full[sbuf]);
        commit_elect(&sb.k_empty[slot]);
        if (s == nsteps - 1) commit_elect(&sb.q_empty);
        if (s > 0 && !issue_pv(step - 1, prev_two, s == 1)) { ok = false; break; }
        prev_two = two;
      }
      if (!ok) break;
      if (!issue_pv(step - 1, prev_two, nsteps == 1)) break;
      commit_elect(&sb.o_full);
    }
    // all issued MMAs complete before TMEM is released
    commit_elect(&sb.final_mma);
    mbar_wait(&sb.final_mma, 0, kWaitNs);
  } else {
    // ===================================================== softmax + epilogue
    const int quarter = warp & 3;                // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;         // tile row 0..127
    const int half = row >> 6;                   // 0: first cube, 1: second cube
    const uint32_t mybit = half ? kSelB : kSelA;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = g.scale * 1.4426950408889634f;  // scale * log2(e)
    uint32_t step = 0;
    int it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < P.n_items && ok && !is_aborted(abort_flag);
         item += gridDim.x) {
      const PairItem pi = P.items[item];
      if (pi.count == 0) continue;
      const uint32_t* list = P.lists + pi.off;
      const int nsteps = (pi.count + 1) / 2;
      float m_run = -INFINITY, l_run = 0.f;
      for (int s = 0; s < nsteps; ++s, ++step) {
        const uint32_t sbuf = step & 1;
        const bool two = 2 * s + 1 < pi.count;
        const bool v0 = (list[2 * s] & mybit) != 0;
        const bool v1 = two && (list[2 * s + 1] & mybit) != 0;
        if (!waitw(&sb.s_full[sbuf], (step >> 1) & 1, abort_flag, P.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ts = tb + lane_addr + kColS + sbuf * 128;
        uint32_t x[128];  // S row; its first 64 words are reused for the packed P
        if (!v0 && !v1) {
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = 0u;
        } else {
          tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
          tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
          if (two) {
            tmem_ld32(ts + 64, *reinterpret_cast<uint32_t(*)[32]>(&x[64]));
            tmem_ld32(ts + 96, *reinterpret_cast<uint32_t(*)[32]>(&x[96]));
          }
          tmem_wait_ld();
          float mx = -INFINITY;
          if (v0) {
#pragma unroll
            for (int i = 0; i < 64; ++i) mx = fmaxf(mx, __uint_as_float(x[i]));
          }
          if (v1) {
#pragma unroll
            for (int i = 64; i < 128; ++i) mx = fmaxf(mx, __uint_as_float(x[i]));
          }
          const float m_new = fmaxf(m_run, mx * c);
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
          if (__any_sync(0xffffffffu, resc)) {
            // O holds the previous steps' sum: wait for the last PV, scale in TMEM
            if (!waitw(&sb.o_ready, (step - 1) & 1, abort_flag, P.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t to = tb + lane_addr + kColO;
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
              uint32_t ov[32];
              tmem_ld32(to + cc, ov);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(to + cc, ov);
            }
            tmem_wait_st();
          }
          float lsum = 0.f;
          const float mb = m_run;
          // x[i] <- bf16x2(p[2i], p[2i+1]); x[2i], x[2i+1] are read before x[i] is written
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const bool valid = (i < 32) ? v0 : v1;
            float p0 = 0.f, p1 = 0.f;
            if (valid) {
              p0 = ex2_approx(fmaf(__uint_as_float(x[2 * i]), c, -mb));
              p1 = ex2_approx(fmaf(__uint_as_float(x[2 * i + 1]), c, -mb));
            }
            lsum += p0 + p1;
            x[i] = pack_f16x2(p0, p1);
          }
          l_run += lsum;
        }
        // P overwrites the first 64 columns of this S buffer (already in registers)
        tmem_st32(ts, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        if (two) tmem_st32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sb.p_full[sbuf]);
      }
      if (!ok) break;
      // ---------------------------------------------- epilogue
      if (!waitw(&sb.o_full, it & 1, abort_flag, P.status)) break;
      ++it;
      tc_fence_after();
      if (half == 0 || pi.b >= 0) {
        const int cube = half ? pi.b : pi.a;
        const int o_in = row & 63;
        const float inv_l = 1.f / l_run;
        const size_t crow = static_cast<size_t>(pi.bh) * g.N + caller_row(g, cube, o_in);
        const size_t frow = static_cast<size_t>(pi.bh) * g.N + cube * kTile + o_in;
        const float* ocr = P.oc + (static_cast<size_t>(pi.bh) * g.Nc + cube) * D;
        const uint32_t to = tb + lane_addr + kColO;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t ov[32];
          tmem_ld32(to + cc, ov);
          tmem_wait_ld();
          float of[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) of[i] = __uint_as_float(ov[i]) * inv_l;
          if (P.o_f) {
            float4* dst = reinterpret_cast<float4*>(P.o_f + frow * D + cc);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(of[4 * i], of[4 * i + 1], of[4 * i + 2], of[4 * i + 3]);
          }
          const uint4* gcp = reinterpret_cast<const uint4*>(P.gc + crow * D + cc);
          const uint4* gfp = reinterpret_cast<const uint4*>(P.gf + crow * D + cc);
          const float4* ocp = reinterpret_cast<const float4*>(ocr + cc);
          uint4* op = reinterpret_cast<uint4*>(P.o + crow * D + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 ga = gcp[v], gb = gfp[v];
            const float4 oa = ocp[2 * v], ob = ocp[2 * v + 1];
            const float ocv[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
            const __nv_bfloat162* g2c = reinterpret_cast<const __nv_bfloat162*>(&ga);
            const __nv_bfloat162* g2f = reinterpret_cast<const __nv_bfloat162*>(&gb);
            uint4 res;
            uint32_t* rp = reinterpret_cast<uint32_t*>(&res);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 fc = __bfloat1622float2(g2c[e]);
              const float2 ff = __bfloat1622float2(g2f[e]);
              const float y0 = fmaf(ocv[2 * e], fc.x, of[8 * v + 2 * e] * ff.x);
              const float y1 = fmaf(ocv[2 * e + 1], fc.y, of[8 * v + 2 * e + 1] * ff.y);
              rp[e] = pack_bf16x2(y0, y1);
            }
            op[v] = res;
          }
        }
        if (P.lse_f) P.lse_f[frow] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tb, kTmemCols);
}

template <int D>
cudaError_t run_fwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                    FwdParams p, cudaStream_t s) {
  alignas(64) CUtensorMap mq, mk, mv;
  const uint64_t rows = static_cast<uint64_t>(g.BH) * g.N;
  if (!encode_tiled_2d(&mq, q, rows, D, 64, 64) || !encode_tiled_2d(&mk, k, rows, D, 64, 64) ||
      !encode_tiled_2d(&mv, v, rows, D, 64, 64))
    return cudaErrorInvalidValue;
  const int smem = FwdSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(fine_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = p.n_items < sms ? p.n_items : sms;
  if (grid <= 0) return cudaSuccess;
  fine_fwd_kernel<D><<<grid, kThreadsFwd, smem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fine_fwd(const Geom& g, const __half* q, const __half* k, const __half* v,
                            const __nv_bfloat16* gc, const __nv_bfloat16* gf, const float* oc,
                            __nv_bfloat16* o, float* o_f, float* lse_f, const Workspace& ws,
                            cudaStream_t s) {
  FwdParams p{g, ws.qpairs, ws.qlist, ws.n_qpairs, gc, gf, oc, o, o_f, lse_f, ws.status};
  if (g.D == 64) return run_fwd<64>(g, q, k, v, p, s);
  return run_fwd<128>(g, q, k, v, p, s);
}

}  // namespace vsa

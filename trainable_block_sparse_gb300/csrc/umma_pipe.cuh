// Helpers shared by the warp-specialised tcgen05 kernels: bounded waits that
// record a time-out and raise a CTA-wide abort flag, and batched UMMA issue
// from a converged warp (one elect per batch; issuing one MMA per elect costs
// about twice the tensor-pipe time of an M=128, N=128, K=16 MMA).
#pragma once

#include <type_traits>

#include "sm103_ptx.cuh"

namespace vsa {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait

// Compile-time loop: f(std::integral_constant<int, i>) for i = 0 .. N-1, so
// the index can select code paths with `if constexpr`.
template <int N, int I = 0, class F>
__device__ __forceinline__ void unroll_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    unroll_for<N, I + 1>(f);
  }
}

__device__ __forceinline__ bool is_aborted(const int* flag) {
  return *reinterpret_cast<const volatile int*>(flag) != 0;
}

__device__ __forceinline__ void raise_abort(int* flag, uint32_t* status) {
  flag_error(status, kDevTimeout);
  *reinterpret_cast<volatile int*>(flag) = 1;
}

// Single-thread bounded wait.
__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, int* flag,
                                      uint32_t* status) {
  if (mbar_wait(bar, parity, kWaitNs)) return true;
  raise_abort(flag, status);
  return false;
}

// Whole-warp bounded wait with a warp-uniform outcome, so the warp stays
// converged for the .sync.aligned tcgen05 operations that follow.
__device__ __forceinline__ bool waitw(uint64_t* bar, uint32_t parity, int* flag,
                                      uint32_t* status) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, kWaitNs));
  if (!ok && (threadIdx.x & 31) == 0) raise_abort(flag, status);
  return ok;
}

// SS chain of kSteps MMAs (K = 16 each), both operands K-major in smem; the
// first MMA overwrites D, the rest accumulate.
template <int kSteps>
__device__ __forceinline__ void issue_ss_chain(uint32_t d_tmem, const uint64_t (&a)[kSteps],
                                               const uint64_t (&b)[kSteps], uint32_t idesc) {
  static_assert(kSteps == 4 || kSteps == 8, "head_dim 64 or 128");
  if constexpr (kSteps == 4) {
    asm volatile(
        "{\n\t.reg .pred p, f, t;\n\telect.sync _|p, 0xffffffff;\n\t"
        "setp.ne.b32 f, %10, %10;\n\tsetp.eq.b32 t, %10, %10;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, f;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, t;\n\t}" ::"r"(d_tmem),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
        "r"(idesc), "r"(0)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, f, t;\n\telect.sync _|p, 0xffffffff;\n\t"
        "setp.ne.b32 f, %18, %18;\n\tsetp.eq.b32 t, %18, %18;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, f;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, t;\n\t}" ::"r"(d_tmem),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
        "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
        "r"(idesc), "r"(0)
        : "memory");
  }
}

// TS chain of 4 MMAs over 64 values of K: A from TMEM (8 columns per 16 K),
// B = 4 smem descriptors.  acc0 = 0 makes the first MMA overwrite D.
__device__ __forceinline__ void issue_ts4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                          uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc,
                                          uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q, t;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %7, 0;\n\t"
      "setp.eq.b32 t, %7, %7;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %6, q;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %3, %6, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %4, %6, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%10], %5, %6, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(acc0), "r"(a_tmem + 8),
      "r"(a_tmem + 16), "r"(a_tmem + 24)
      : "memory");
}

// D (+)= A[tmem, 128 x 64*ntiles] * B[smem, MN-major rows of 128 bytes]: the
// B stage holds 128 K-rows per 64-wide N chunk, K-steps of 16 rows = 2048 bytes.
// The packed A columns of the second 64 values of K start `a_second` columns
// after those of the first.
__device__ __forceinline__ void issue_ts_rows(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              bool two, uint32_t idesc, bool accumulate,
                                              uint32_t a_second = 32) {
  issue_ts4(d_tmem, a_tmem, b_desc, b_desc + (2048 >> 4), b_desc + (4096 >> 4),
            b_desc + (6144 >> 4), idesc, accumulate ? 1u : 0u);
  if (two)
    issue_ts4(d_tmem, a_tmem + a_second, b_desc + (8192 >> 4), b_desc + (10240 >> 4),
              b_desc + (12288 >> 4), b_desc + (14336 >> 4), idesc, 1u);
}

// e4m3 SS chain of 4 MMAs (K = 32 each, 128 values of K), both operands
// K-major in smem; the first MMA overwrites D.
__device__ __forceinline__ void issue_ss4_f8(uint32_t d_tmem, const uint64_t (&a)[4],
                                             const uint64_t (&b)[4], uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p, f, t;\n\telect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 f, %10, %10;\n\tsetp.eq.b32 t, %10, %10;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %5, %9, f;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %6, %9, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %7, %9, t;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %8, %9, t;\n\t}" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
      "r"(idesc), "r"(0)
      : "memory");
}

// e4m3 TS chain over 64 values of K: A from TMEM (8 columns, four e4m3 per
// column, per 32 K), B = 2 smem descriptors.  acc0 = 0: the first MMA
// overwrites D.
__device__ __forceinline__ void issue_ts2_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                             uint64_t b1, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q, t;\n\telect.sync _|p, 0xffffffff;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "setp.eq.b32 t, %5, %5;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %4, q;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%6], %3, %4, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b0), "l"(b1), "r"(idesc), "r"(acc0), "r"(a_tmem + 8)
      : "memory");
}

// Per-warpgroup register split (every warp of a warpgroup executes the same
// one; the increases and decreases of a block must add up within the
// registers it was launched with).
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

}  // namespace vsa

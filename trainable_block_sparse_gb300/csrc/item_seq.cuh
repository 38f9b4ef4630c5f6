// Dynamic item schedule of the persistent fine kernels.
//
// The kernels walk a list of work items (query-cube pairs, or key-cube pairs
// in the key-major backward pass) in a fixed schedule order.  Rather than
// CTA b taking positions b, b + grid, ... (which leaves the CTAs' totals of
// tile steps a few percent apart, and the kernel as long as the largest),
// one thread of each CTA takes the next position from a per-launch counter in
// global memory (atomicAdd: every position goes to exactly one CTA) whenever
// its CTA has room for another item, so the CTAs finish within about one item
// of each other.  Positions are still taken in schedule order, so the items
// running at any moment stay neighbours (sharing K/V tiles in L2), and every
// item is computed by one CTA alone, so results do not depend on which CTA
// takes it.
//
// Within the CTA the fetcher publishes the positions, in the order taken,
// through a ring of kSeqSlots shared-memory slots; every role (each producer
// thread, the UMMA warp, each softmax and epilogue warp) reads the same
// sequence and releases each slot after reading it.  All waits are bounded.
#pragma once

#include "umma_pipe.cuh"

namespace vsa {

constexpr int kSeqSlots = 4;
constexpr int kSeqEnd = -1;    // the schedule is exhausted
constexpr int kSeqAbort = -2;  // a wait timed out (the CTA's abort flag is raised)

struct ItemSeq {
  uint64_t full[kSeqSlots];   // one arrival: the fetcher has published the slot
  uint64_t empty[kSeqSlots];  // one arrival per consumer: all have read it
  int pos[kSeqSlots];
};

// One thread, before the CTA-wide barrier that follows barrier set-up.
__device__ __forceinline__ void seq_init(ItemSeq& q, uint32_t consumers) {
  for (int i = 0; i < kSeqSlots; ++i) {
    mbar_init(&q.full[i], 1);
    mbar_init(&q.empty[i], consumers);
  }
}

// Fetcher (one thread): schedule positions from the launch's counter (zero at
// launch), published in the order taken, until the first position past the
// last item, which is published as kSeqEnd.
__device__ __forceinline__ void seq_fetch(ItemSeq& q, int* counter, int n_items, int* abort_flag,
                                          uint32_t* status) {
  for (uint32_t s = 0;; ++s) {
    const uint32_t slot = s % kSeqSlots;
    if (s >= kSeqSlots &&
        !wait1(&q.empty[slot], ((s / kSeqSlots) & 1) ^ 1, abort_flag, status))
      return;
    const int p = is_aborted(abort_flag) ? n_items : atomicAdd(counter, 1);
    q.pos[slot] = p < n_items ? p : kSeqEnd;
    mbar_arrive(&q.full[slot]);  // release: a consumer's wait acquires pos
    if (p >= n_items) return;
  }
}

// The next schedule position for one consumer (kSeqEnd at the end, kSeqAbort
// after a time-out); `s` counts the entries this consumer has read.  A warp
// consumer calls it with all 32 lanes and arrives once; a single-thread
// consumer (a producer lane) passes kWarp = false.
template <bool kWarp>
__device__ __forceinline__ int seq_next(ItemSeq& q, uint32_t& s, int* abort_flag,
                                        uint32_t* status) {
  const uint32_t slot = s % kSeqSlots, parity = (s / kSeqSlots) & 1;
  const bool ok = kWarp ? waitw(&q.full[slot], parity, abort_flag, status)
                        : wait1(&q.full[slot], parity, abort_flag, status);
  if (!ok) return kSeqAbort;
  const int p = *reinterpret_cast<volatile const int*>(&q.pos[slot]);
  if (kWarp) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&q.empty[slot]);
  } else {
    mbar_arrive(&q.empty[slot]);
  }
  ++s;
  return p;
}

// The position `ahead` entries past a warp consumer's next one, without
// reading it off.  ahead <= kSeqSlots - 2 never makes the fetcher wait for
// this consumer: the slot it needs was released with entries this consumer
// has already read.
__device__ __forceinline__ int seq_peek(ItemSeq& q, uint32_t s, int ahead, int* abort_flag,
                                        uint32_t* status) {
  const uint32_t e = s + static_cast<uint32_t>(ahead);
  const uint32_t slot = e % kSeqSlots, parity = (e / kSeqSlots) & 1;
  if (!waitw(&q.full[slot], parity, abort_flag, status)) return kSeqAbort;
  return *reinterpret_cast<volatile const int*>(&q.pos[slot]);
}

}  // namespace vsa

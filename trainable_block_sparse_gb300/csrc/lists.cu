// Work lists for the block-sparse kernels.
//
// The fine stage runs 128-row tensor-core tiles, i.e. two 64-token query cubes
// at a time; a pair iterates over the union of its two index lists, and a bit
// per entry says which of the two cubes selected that key cube (rows of the
// other cube see the tile as masked).  The backward pass over keys needs the
// transposed relation (for each key cube, the query cubes that selected it),
// and pairs key cubes the same way.
//
// Every list entry read here is range-checked: an id outside [0, Nc), a list
// that is not strictly ascending, or a count outside [1, capacity] sets
// kDevBadIndex in the status word and the offending entry is dropped, so no
// later kernel ever addresses memory outside the tensors.
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

__device__ __forceinline__ int checked_count(const Geom& g, const int* cnt, size_t row,
                                             uint32_t* status) {
  int c = cnt[row];
  if (c < 1 || c > g.cap) {
    flag_error(status, kDevBadIndex);
    c = min(max(c, 0), g.cap);
  }
  return c;
}

// Sorted merge of two ascending lists into `out`, tagging each entry.
__device__ int merge_lists(const int* la, int ca, const int* lb, int cb, int limit,
                           uint32_t* out, uint32_t* status) {
  int i = 0, j = 0, n = 0, prev = -1;
  while (i < ca || j < cb) {
    const int va = i < ca ? la[i] : 0x7fffffff;
    const int vb = j < cb ? lb[j] : 0x7fffffff;
    int v;
    uint32_t f;
    if (va == vb) { v = va; f = kSelA | kSelB; ++i; ++j; }
    else if (va < vb) { v = va; f = kSelA; ++i; }
    else { v = vb; f = kSelB; ++j; }
    if (v < 0 || v >= limit || v <= prev) {
      flag_error(status, kDevBadIndex);
      continue;
    }
    prev = v;
    out[n++] = static_cast<uint32_t>(v) | f;
  }
  return n;
}

__global__ void build_qpairs_kernel(Geom g, const int* __restrict__ idx,
                                    const int* __restrict__ cnt, Workspace ws) {
  const int npb = (g.Nc + 1) / 2;
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= g.BH * npb) return;
  const int bh = item / npb, p = item % npb;
  const int a = 2 * p, b = (2 * p + 1 < g.Nc) ? 2 * p + 1 : -1;
  const size_t ra = static_cast<size_t>(bh) * g.Nc + a;
  const int ca = checked_count(g, cnt, ra, ws.status);
  int cb = 0;
  const int* lb = nullptr;
  if (b >= 0) {
    cb = checked_count(g, cnt, ra + 1, ws.status);
    lb = idx + (ra + 1) * g.cap;
  }
  const int off = item * 2 * g.cap;
  const int n = merge_lists(idx + ra * g.cap, ca, lb, cb, g.Nc, ws.qlist + off, ws.status);
  ws.qpairs[item] = PairItem{bh, a, b, n, off};
}

// Selection bit matrix: row i (query cube) has bit j set when j is in its list.
__global__ void build_mask_kernel(Geom g, const int* __restrict__ idx,
                                  const int* __restrict__ cnt, Workspace ws) {
  const int words = (g.Nc + 31) / 32;
  const size_t row = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= static_cast<size_t>(g.BH) * g.Nc) return;
  uint32_t* m = ws.tmask + row * words;
  for (int w = 0; w < words; ++w) m[w] = 0u;
  const int c = checked_count(g, cnt, row, ws.status);
  const int* l = idx + row * g.cap;
  for (int e = 0; e < c; ++e) {
    const int j = l[e];
    if (j < 0 || j >= g.Nc) {
      flag_error(ws.status, kDevBadIndex);
      continue;
    }
    m[j >> 5] |= 1u << (j & 31);
  }
}

// Transposed lists: for key cube j of a (batch, head), the ascending query
// cubes whose selection bit j is set.  Three small kernels, each over
// (batch*head) x (32-cube columns of the bit matrix) or per (batch*head):
//   count: per key cube, how many query cubes selected it;
//   scan:  exclusive prefix of the counts = CSR offsets;
//   fill:  each warp of the CTA takes a contiguous range of query cubes, so
//          the entries of each key cube come out in ascending order.
constexpr int kTransposeWarps = 8;

// Per-warp counts of bit (lane) of column word w over the warp's row range.
__device__ __forceinline__ int column_count(const uint32_t* m, int words, int w, int i0, int i1) {
  const int lane = threadIdx.x & 31;
  int c = 0;
  for (int i = i0; i < i1; ++i) c += (m[static_cast<size_t>(i) * words + w] >> lane) & 1u;
  return c;
}

__global__ void __launch_bounds__(kTransposeWarps * 32) transpose_count_kernel(Geom g, Workspace ws) {
  __shared__ int part[kTransposeWarps][32];
  const int bh = blockIdx.x, w = blockIdx.y;
  const int words = (g.Nc + 31) / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int chunk = (g.Nc + kTransposeWarps - 1) / kTransposeWarps;
  const int i0 = min(warp * chunk, g.Nc), i1 = min(i0 + chunk, g.Nc);
  const uint32_t* m = ws.tmask + static_cast<size_t>(bh) * g.Nc * words;
  part[warp][lane] = column_count(m, words, w, i0, i1);
  __syncthreads();
  if (warp == 0) {
    int c = 0;
    for (int k = 0; k < kTransposeWarps; ++k) c += part[k][lane];
    const int j = 32 * w + lane;
    if (j < g.Nc) ws.toff[static_cast<size_t>(bh) * (g.Nc + 1) + j + 1] = c;
  }
}

// In-place inclusive scan of toff[1..Nc] (holding counts) with toff[0] = 0.
__global__ void __launch_bounds__(1024) transpose_scan_kernel(Geom g, Workspace ws) {
  __shared__ int wsum[32];
  int* toff = ws.toff + static_cast<size_t>(blockIdx.x) * (g.Nc + 1);
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int carry = 0;
  for (int base = 0; base < g.Nc; base += blockDim.x) {
    const int j = base + threadIdx.x;
    int v = j < g.Nc ? toff[j + 1] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += u;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int x = lane < static_cast<int>(blockDim.x / 32) ? wsum[lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += u;
      }
      wsum[lane] = x;  // inclusive prefix over warps
    }
    __syncthreads();
    const int total = wsum[blockDim.x / 32 - 1];
    if (warp > 0) v += wsum[warp - 1];
    if (j < g.Nc) toff[j + 1] = carry + v;
    carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) toff[0] = 0;
}

__global__ void __launch_bounds__(kTransposeWarps * 32) transpose_fill_kernel(Geom g, Workspace ws) {
  __shared__ int part[kTransposeWarps][32];
  const int bh = blockIdx.x, w = blockIdx.y;
  const int words = (g.Nc + 31) / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int chunk = (g.Nc + kTransposeWarps - 1) / kTransposeWarps;
  const int i0 = min(warp * chunk, g.Nc), i1 = min(i0 + chunk, g.Nc);
  const uint32_t* m = ws.tmask + static_cast<size_t>(bh) * g.Nc * words;
  part[warp][lane] = column_count(m, words, w, i0, i1);
  __syncthreads();
  const int j = 32 * w + lane;
  if (j >= g.Nc) return;
  int n = ws.toff[static_cast<size_t>(bh) * (g.Nc + 1) + j];
  for (int k = 0; k < warp; ++k) n += part[k][lane];
  int* tl = ws.tlist + static_cast<size_t>(bh) * g.Nc * g.cap;
  for (int i = i0; i < i1; ++i)
    if ((m[static_cast<size_t>(i) * words + w] >> lane) & 1u) tl[n++] = i;
}

__global__ void build_kpairs_kernel(Geom g, Workspace ws) {
  const int npb = (g.Nc + 1) / 2;
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= g.BH * npb) return;
  const int bh = item / npb, p = item % npb;
  const int a = 2 * p, b = (2 * p + 1 < g.Nc) ? 2 * p + 1 : -1;
  const int* toff = ws.toff + static_cast<size_t>(bh) * (g.Nc + 1);
  const int* tl = ws.tlist + static_cast<size_t>(bh) * g.Nc * g.cap;
  const int ca = toff[a + 1] - toff[a];
  const int cb = b >= 0 ? toff[b + 1] - toff[b] : 0;
  const int off = bh * g.Nc * g.cap + toff[a];
  const int n = merge_lists(tl + toff[a], ca, b >= 0 ? tl + toff[b] : nullptr, cb, g.Nc,
                            ws.klist + off, ws.status);
  ws.kpairs[item] = PairItem{bh, a, b, n, off};
}

// ---------------------------------------------------------- item schedule
// Steps of an item = ceil(|union| / 2) <= 256; key index 0 = most steps.
constexpr int kOrderKeys = 264;

__device__ __forceinline__ int order_key(const PairItem& it) {
  const int steps = min((it.count + 1) / 2, kOrderKeys - 1);
  return kOrderKeys - 1 - steps;
}

__global__ void order_count_kernel(const PairItem* __restrict__ items, int n, int* hist) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) atomicAdd(&hist[order_key(items[i])], 1);
}

// hist -> exclusive prefix (bucket starts), one warp.
__global__ void order_scan_kernel(int* hist) {
  const int lane = threadIdx.x;
  int carry = 0;
  for (int base = 0; base < kOrderKeys; base += 32) {
    const int k = base + lane;
    const int v = k < kOrderKeys ? hist[k] : 0;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += u;
    }
    if (k < kOrderKeys) hist[k] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Items into their buckets, largest first (order within a bucket is
// arbitrary: it only decides which CTA runs an item, never what the item
// computes).  The kernels' CTAs take positions from a shared counter as they
// free up, so largest-first is the longest-processing-time rule.
__global__ void order_scatter_kernel(const PairItem* __restrict__ items, int n, int* cursor,
                                     int* sorted) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) sorted[atomicAdd(&cursor[order_key(items[i])], 1)] = i;
}

}  // namespace

int persistent_grid(int n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return n < sms ? n : sms;
}

cudaError_t launch_item_order(const PairItem* items, int n, int* order, int* tmp,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int* hist = tmp;
  cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(int) * kOrderKeys, s);
  if (e != cudaSuccess) return e;
  const int blocks = (n + 255) / 256;
  order_count_kernel<<<blocks, 256, 0, s>>>(items, n, hist);
  order_scan_kernel<<<1, 32, 0, s>>>(hist);
  order_scatter_kernel<<<blocks, 256, 0, s>>>(items, n, hist, order);
  return cudaGetLastError();
}

cudaError_t launch_build_qpairs(const Geom& g, const int* idx, const int* cnt,
                                const Workspace& ws, cudaStream_t s) {
  const int items = g.BH * ((g.Nc + 1) / 2);
  build_qpairs_kernel<<<(items + 127) / 128, 128, 0, s>>>(g, idx, cnt, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !ws.qorder || !use_cost_order(g)) return e;
  return launch_item_order(ws.qpairs, items, ws.qorder, ws.order_tmp, s);
}

cudaError_t launch_build_kpairs(const Geom& g, const int* idx, const int* cnt,
                                const Workspace& ws, cudaStream_t s) {
  const size_t rows = static_cast<size_t>(g.BH) * g.Nc;
  build_mask_kernel<<<static_cast<unsigned>((rows + 127) / 128), 128, 0, s>>>(g, idx, cnt, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid(g.BH, (g.Nc + 31) / 32);
  transpose_count_kernel<<<grid, kTransposeWarps * 32, 0, s>>>(g, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  transpose_scan_kernel<<<g.BH, 1024, 0, s>>>(g, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  transpose_fill_kernel<<<grid, kTransposeWarps * 32, 0, s>>>(g, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int items = g.BH * ((g.Nc + 1) / 2);
  build_kpairs_kernel<<<(items + 127) / 128, 128, 0, s>>>(g, ws);
  if ((e = cudaGetLastError()) != cudaSuccess || !ws.korder || !use_cost_order(g)) return e;
  return launch_item_order(ws.kpairs, items, ws.korder, ws.order_tmp, s);
}

}  // namespace vsa

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

// Transposed lists of one (batch, head): for key cube j, the ascending query
// cubes whose bit j is set.  One CTA per (batch, head).
__global__ void __launch_bounds__(1024) build_transpose_kernel(Geom g, Workspace ws) {
  extern __shared__ int offs[];  // [Nc + 1]
  const int bh = blockIdx.x;
  const int words = (g.Nc + 31) / 32;
  const uint32_t* m = ws.tmask + static_cast<size_t>(bh) * g.Nc * words;
  for (int j = threadIdx.x; j < g.Nc; j += blockDim.x) {
    int c = 0;
    const uint32_t bit = 1u << (j & 31);
    for (int i = 0; i < g.Nc; ++i) c += (m[static_cast<size_t>(i) * words + (j >> 5)] & bit) != 0;
    offs[j + 1] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    offs[0] = 0;
    for (int j = 0; j < g.Nc; ++j) offs[j + 1] += offs[j];
  }
  __syncthreads();
  int* toff = ws.toff + static_cast<size_t>(bh) * (g.Nc + 1);
  int* tl = ws.tlist + static_cast<size_t>(bh) * g.Nc * g.cap;
  for (int j = threadIdx.x; j <= g.Nc; j += blockDim.x) toff[j] = offs[j];
  for (int j = threadIdx.x; j < g.Nc; j += blockDim.x) {
    int n = offs[j];
    const uint32_t bit = 1u << (j & 31);
    for (int i = 0; i < g.Nc; ++i)
      if (m[static_cast<size_t>(i) * words + (j >> 5)] & bit) tl[n++] = i;
  }
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

}  // namespace

cudaError_t launch_build_qpairs(const Geom& g, const int* idx, const int* cnt,
                                const Workspace& ws, cudaStream_t s) {
  const int items = g.BH * ((g.Nc + 1) / 2);
  build_qpairs_kernel<<<(items + 127) / 128, 128, 0, s>>>(g, idx, cnt, ws);
  return cudaGetLastError();
}

cudaError_t launch_build_kpairs(const Geom& g, const int* idx, const int* cnt,
                                const Workspace& ws, cudaStream_t s) {
  const size_t rows = static_cast<size_t>(g.BH) * g.Nc;
  build_mask_kernel<<<static_cast<unsigned>((rows + 127) / 128), 128, 0, s>>>(g, idx, cnt, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(int) * (g.Nc + 1);
  build_transpose_kernel<<<g.BH, 1024, smem, s>>>(g, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int items = g.BH * ((g.Nc + 1) / 2);
  build_kpairs_kernel<<<(items + 127) / 128, 128, 0, s>>>(g, ws);
  return cudaGetLastError();
}

}  // namespace vsa

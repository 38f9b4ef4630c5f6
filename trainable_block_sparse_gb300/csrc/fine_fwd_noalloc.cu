// vsa_fine_fwd_noalloc: the fine stage + combine of vsa_fine_fwd for callers
// that cannot hand the library a scratch buffer.
//
// Some callers hold no device allocator of their own: a plugin run by a host
// engine that owns all device memory and gives the plugin only its input and
// output buffers, or a fixed-footprint runtime that reserves every byte before
// it starts.  Such a caller cannot call cudaMalloc and cannot provide the `ws`
// buffer the other entry points take.  This variant keeps its scratch (the
// status word, the query-pair work items and their union lists) in a
// fixed-size array in device memory that belongs to the library itself.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoallocScratchBytes until the process exits.  Host code
// cannot pass the array's name to a kernel (on the host the name is only a
// stand-in, not a device address), so the first call on each device, with that
// device current, looks the device address up with cudaGetSymbolAddress and
// caches it; make that first call before any stream capture.  Every call shares
// the one array, so calls that overlap on the GPU race with each other; the
// status word is cleared at the start of each call, the rest is fully
// rewritten before it is read.  The query pairs run in their natural order
// (the cost-sorted order of vsa_fine_fwd would need more scratch); results are
// bitwise those of vsa_fine_fwd.
#include <mutex>

#include "../../include/vsa.h"
#include "sm103_ptx.cuh"
#include "vsa_common.cuh"

namespace vsa {
namespace {

constexpr size_t kNoallocScratchBytes = VSA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" vsa_status_t vsa_fine_fwd_noalloc(const vsa_config_t* cfg, const void* q16,
                                             const void* k16, const void* v16,
                                             const int32_t* idx, const int32_t* cnt,
                                             const void* gc, const void* gf, const float* oc,
                                             void* o, void* o_f, float* lse_f,
                                             uint32_t* status, void* stream) {
  Geom g;
  const vsa_status_t st = make_geom(cfg, &g);
  if (st != VSA_OK) return st;
  // scratch: status word, schedule counters (in the first 256 bytes) | pair
  // items | union lists (2 * capacity entries per pair)
  const size_t npairs = static_cast<size_t>(g.BH) * ((g.Nc + 1) / 2);
  const size_t items_off = 256;
  const size_t lists_off = items_off + round256(sizeof(PairItem) * npairs);
  const size_t need = lists_off + round256(sizeof(uint32_t) * npairs * 2 * g.cap);
  if (need > kNoallocScratchBytes) return VSA_ERR_SHAPE;  // beyond the fixed scratch array
  if (!q16 || !k16 || !v16 || !idx || !cnt || !gc || !gf || !oc || !o) return VSA_ERR_INVALID_ARG;
  if (!aligned(q16) || !aligned(k16) || !aligned(v16) || !aligned(idx) || !aligned(cnt) ||
      !aligned(gc) || !aligned(gf) || !aligned(oc) || !aligned(o) || !aligned(o_f) ||
      !aligned(lse_f) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return VSA_ERR_ALIGNMENT;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return VSA_ERR_CUDA;
  char* b = static_cast<char*>(base);
  Workspace w{};
  w.status = reinterpret_cast<uint32_t*>(b);
  w.counter = reinterpret_cast<int*>(b + 64);
  w.qpairs = reinterpret_cast<PairItem*>(b + items_off);
  w.qlist = reinterpret_cast<uint32_t*>(b + lists_off);
  w.n_qpairs = static_cast<int>(npairs);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(w.status, 0, sizeof(uint32_t), s) != cudaSuccess) return VSA_ERR_CUDA;
  if (launch_build_qpairs(g, idx, cnt, w, s) != cudaSuccess) return VSA_ERR_CUDA;
  if (launch_fine_fwd(g, static_cast<const __half*>(q16), static_cast<const __half*>(k16),
                      static_cast<const __half*>(v16), static_cast<const __nv_bfloat16*>(gc),
                      static_cast<const __nv_bfloat16*>(gf), oc, static_cast<__nv_bfloat16*>(o),
                      static_cast<__half*>(o_f), lse_f, w, s) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (status &&
      cudaMemcpyAsync(status, w.status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return VSA_ERR_CUDA;
  return VSA_OK;
}

// rkv_decode_attn_static: decode attention whose split-K partials live in a
// fixed array inside the library, so the call allocates nothing.
//
// Who needs it: code that may not allocate device memory at the point where
// it runs attention.  A real-time audio callback has a clock-step budget of
// 80 ms and cannot afford an allocator call that may synchronise the device;
// a plug-in hosted by a serving engine whose caching allocator has already
// reserved the free HBM has no memory of its own to ask for.  Such callers
// pass only inputs and outputs here; the partial results of a window split
// over several CTAs go to the array below, which every process that loads the
// library holds on every device it uses until exit.  A call whose windows are
// not split writes its outputs directly and touches the array not at all.
#include <mutex>

#include "rkv_internal.cuh"

namespace rkv {
namespace {

// 8 MiB of fp32 partials: (m, l) and head_dim outputs per (active stream, query row, split).
constexpr size_t kStaticScratchFloats = size_t(2) << 20;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device with that device current.  In host code the array's name is only a
// stand-in; kernels must be given this address.
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

// Partial rows of one call: one per (active stream, query row, split), none when the plan
// does not split the windows (the kernel then writes out and lse itself).
size_t partial_rows(const AttnPlan& p, const DevView& v, int n_active) {
  if (p.splits <= 1) return 0;
  return static_cast<size_t>(n_active) * v.q_per_step * v.n_q_heads * p.splits;
}

size_t ml_floats(size_t rows) {
  return (rows * 2 + 63) / 64 * 64;  // keeps the outputs that follow 256-byte aligned
}

}  // namespace

size_t static_scratch_floats() { return kStaticScratchFloats; }

size_t static_scratch_need(const DevView& v, int n_active) {
  const size_t rows = partial_rows(plan_decode_attn(v, n_active, 1, false), v, n_active);
  return rows == 0 ? 0 : ml_floats(rows) + rows * v.head_dim;
}

cudaError_t launch_decode_attn_static(const DevView& v, int n_active, int layer, const uint16_t* q, uint16_t* out,
                                      float* lse, cudaStream_t st) {
  float* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return e;
  const size_t rows = partial_rows(plan_decode_attn(v, n_active, 1, false), v, n_active);
  DevView w = v;
  w.part_ml = base;
  w.part_o = base + ml_floats(rows);
  return launch_decode_attn_scratch(w, n_active, layer, q, out, lse, st);
}

}  // namespace rkv

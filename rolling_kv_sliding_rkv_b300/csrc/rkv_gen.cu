// Counter-based synthetic inputs on the device.
//
// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): z += golden increment; z = (z ^ z>>30) * M1;
// z = (z ^ z>>27) * M2; z ^= z>>31.  A token's key is the chain
// sm(sm(sm(sm(sm(seed) ^ tag) ^ stream) ^ layer) ^ token); element e uses the
// words sm(key + 3e + r), r < 3, four 12-bit fields each.  The twelve fields
// sum to S and x = (S - 24570) / 4096 (exact in fp32, mean 0, variance ~1);
// the output is bf16_rne(fp32(x) * scale).  Integer arithmetic, one fp32
// multiply and one rounding: the host generator produces the same bits.
#include "rkv_internal.cuh"

namespace rkv {
namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t token_key(uint64_t seed, uint32_t tag, int32_t stream, int32_t layer,
                                              int64_t token) {
  uint64_t k = splitmix64(seed);
  k = splitmix64(k ^ static_cast<uint64_t>(tag));
  k = splitmix64(k ^ static_cast<uint64_t>(static_cast<int64_t>(stream)));
  k = splitmix64(k ^ static_cast<uint64_t>(static_cast<int64_t>(layer)));
  return splitmix64(k ^ static_cast<uint64_t>(token));
}

__device__ __forceinline__ uint16_t draw(uint64_t key, int64_t e, float scale) {
  int32_t total = 0;
  const uint64_t base = key + 3ull * static_cast<uint64_t>(e);
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const uint64_t w = splitmix64(base + r);
#pragma unroll
    for (int f = 0; f < 4; ++f) total += static_cast<int32_t>((w >> (12 * f)) & 0xFFFu);
  }
  const float x = static_cast<float>(total - 24570) / 4096.0f;  // exact
  return f32_to_bf16(__fmul_rn(x, scale));
}

__global__ void gen_tokens_kernel(uint64_t seed, uint32_t tag, int32_t stream, int32_t layer, int64_t token0,
                                  int32_t width, float scale, uint16_t* __restrict__ out) {
  const int t = blockIdx.y;
  const uint64_t key = token_key(seed, tag, stream, layer, token0 + t);
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < width; e += gridDim.x * blockDim.x)
    out[static_cast<int64_t>(t) * width + e] = draw(key, e, scale);
}

// grid (A * Q, 3): tensor 0 = q [A][Q][Hq][d], 1 = k, 2 = v [A][Q][Hkv][d].  Launched with
// programmatic dependent launch and letting its dependents start before it writes, as a
// caller's own kernel that produces the queries of a layer may be.
__global__ void gen_step_kernel(DevView v, uint64_t seed, int32_t layer, float scale, uint16_t* __restrict__ q,
                                uint16_t* __restrict__ k, uint16_t* __restrict__ vv) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x;
  const int a = row / v.q_per_step, t = row % v.q_per_step;
  const int which = blockIdx.y;
  const StepDesc dsc = v.desc[a];
  const int heads = which == 0 ? v.n_q_heads : v.n_kv_heads;
  const int width = heads * v.head_dim;
  uint16_t* dst = (which == 0 ? q : which == 1 ? k : vv) + static_cast<int64_t>(row) * width;
  const uint64_t key = token_key(seed, static_cast<uint32_t>(which + 1), dsc.stream, layer, dsc.n_old + t);
  for (int e = threadIdx.x; e < width; e += blockDim.x) dst[e] = draw(key, e, scale);
}

// The inputs of the next step of the listed streams, all layers: grid (A * Q, 3, L), token
// index = the stream's token count before that step (read from the device state).
__global__ void gen_next_kernel(DevView v, ActiveIds ids, uint64_t seed, float scale, uint16_t* __restrict__ q,
                                uint16_t* __restrict__ k, uint16_t* __restrict__ vv) {
  const int row = blockIdx.x;
  const int a = row / v.q_per_step, t = row % v.q_per_step;
  const int which = blockIdx.y, layer = blockIdx.z;
  const int s = ids.id[a];
  const int64_t n = v.state[static_cast<int64_t>(s) * kStateFields + F_N];
  const int heads = which == 0 ? v.n_q_heads : v.n_kv_heads;
  const int width = heads * v.head_dim;
  const int64_t rows = static_cast<int64_t>(ids.n) * v.q_per_step;
  uint16_t* dst = (which == 0 ? q : which == 1 ? k : vv) + (layer * rows + row) * width;
  const uint64_t key = token_key(seed, static_cast<uint32_t>(which + 1), s, layer, n + t);
  for (int e = threadIdx.x; e < width; e += blockDim.x) dst[e] = draw(key, e, scale);
}

}  // namespace

cudaError_t launch_gen_next_inputs(const DevView& v, const ActiveIds& ids, uint64_t seed, float scale, uint16_t* q,
                                   uint16_t* k, uint16_t* vv, cudaStream_t st) {
  gen_next_kernel<<<dim3(ids.n * v.q_per_step, 3, v.n_layers), 256, 0, st>>>(v, ids, seed, scale, q, k, vv);
  return cudaGetLastError();
}

cudaError_t launch_gen_tokens(uint64_t seed, uint32_t tag, int32_t stream_id, int32_t layer, int64_t token0,
                              int32_t n_tokens, int32_t width, float scale, uint16_t* out, cudaStream_t st) {
  if (n_tokens == 0 || width == 0) return cudaSuccess;
  const int bx = (width + 255) / 256 < 64 ? (width + 255) / 256 : 64;
  gen_tokens_kernel<<<dim3(bx, n_tokens), 256, 0, st>>>(seed, tag, stream_id, layer, token0, width, scale, out);
  return cudaGetLastError();
}

cudaError_t launch_gen_step_inputs(const DevView& v, int n_active, uint64_t seed, int32_t layer, float scale,
                                   uint16_t* q, uint16_t* k, uint16_t* vv, cudaStream_t st) {
  return launch_pdl(gen_step_kernel, dim3(n_active * v.q_per_step, 3), dim3(256), 0, st, v, seed, layer, scale, q, k,
                    vv);
}

}  // namespace rkv

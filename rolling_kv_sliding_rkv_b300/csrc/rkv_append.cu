// RoPE + append (voxtral.c rolling-KV article §二: RoPE is baked into K when
// it is written) and the exact re-base (Audio8 ASR Infinite 无限长转写原理,
// "Rolling KV Cache 三步拆解", 第 2 步: on every roll all retained keys are
// rotated back by the evicted offset, with a strict rotation).
//
// Pairs are (x_i, x_{i+d/2}); (a, b) -> (a cos - b sin, a sin + b cos) in
// fp32.  The rotated key is stored as fp16 (nearest even): eleven significant
// bits keep the score error of a stored key near 2e-4 for unit-variance
// inputs, where bf16 storage would give ~1.6e-3 (the voxtral.c article, §七,
// mentions an fp16 KV cache).  Values and pre-RoPE keys are stored as the
// bf16 inputs, bit for bit.
#include "rkv_internal.cuh"

namespace rkv {
namespace {

constexpr int kWarps = 4;

// One warp per (active stream, new token, kv head): rotate k with the
// token's cos/sin, write it and v into the token's ring slot (and the
// pre-RoPE k in the exact scheme).
__global__ void __launch_bounds__(kWarps * 32) append_rope_kernel(DevView v, int layer, const uint16_t* __restrict__ k,
                                                                  const uint16_t* __restrict__ val) {
  const int row = blockIdx.x;  // a * Q + t
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.y * kWarps + warp;
  const int hkv = v.n_kv_heads, d = v.head_dim, half = d / 2;
  if (kvh >= hkv) return;
  const int a = row / v.q_per_step, t = row % v.q_per_step;
  const float* cs = v.cs_new + static_cast<int64_t>(row) * half * 2;
  const StepDesc dsc = v.desc[a];
  const int64_t tok = dsc.n_old + t;
  const int slot = static_cast<int>(tok % dsc.window);
  const int ring_page = slot / v.page_size;
  if (ring_page >= v.max_pages) {
    if (lane == 0) record_error(v.status, DEV_BOUNDS, 1, ring_page);
    return;
  }
  const int page = v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + ring_page];
  if (page < 0 || page >= v.n_pages) {
    if (lane == 0) record_error(v.status, DEV_BOUNDS, 2, page);
    return;
  }
  const int64_t dst = pool_offset(v, layer, page, kvh, slot % v.page_size);
  const int64_t src = (static_cast<int64_t>(row) * hkv + kvh) * d;
  for (int i = lane; i < half; i += 32) {
    const float c = cs[2 * i], s = cs[2 * i + 1];
    const uint16_t ra = k[src + i], rb = k[src + i + half];
    const float xa = bf16_to_f32(ra), xb = bf16_to_f32(rb);
    const float ya = xa * c - xb * s, yb = xa * s + xb * c;
    if (!fits_f16(ya) || !fits_f16(yb)) record_error(v.status, DEV_RANGE, 1, i);
    v.k_rot[dst + i] = f32_to_f16(ya);
    v.k_rot[dst + i + half] = f32_to_f16(yb);
    if (v.k_raw) {
      v.k_raw[dst + i] = ra;
      v.k_raw[dst + i + half] = rb;
    }
    v.v[dst + i] = val[src + i];
    v.v[dst + i + half] = val[src + i + half];
  }
}

// Grid (active stream, ring page, kv head).  For a stream that re-bases this
// step, every retained key written before the step (tokens evicted ..
// n_old - 1) becomes R(j - rope_base) applied to its pre-RoPE copy: the
// exact result of rotating the previously stored key by R(-delta), with one
// rounding however many re-bases the key has seen.
__global__ void __launch_bounds__(128) rebase_kernel(DevView v, int layer) {
  const int a = blockIdx.x, ring_page = blockIdx.y, kvh = blockIdx.z;
  const StepDesc dsc = v.desc[a];
  if (dsc.delta == 0) return;
  const int ps = v.page_size, d = v.head_dim, half = d / 2;
  const int slot0 = ring_page * ps;
  if (slot0 >= dsc.window) return;
  const int n_slots = min(ps, dsc.window - slot0);
  const int page = v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + ring_page];
  if (page < 0 || page >= v.n_pages) {
    if (threadIdx.x == 0) record_error(v.status, DEV_BOUNDS, 3, page);
    return;
  }
  const int64_t base = pool_offset(v, layer, page, kvh, 0);
  for (int e = threadIdx.x; e < n_slots * half; e += blockDim.x) {
    const int off = e / half, i = e % half;
    const int64_t tok = token_in_slot(slot0 + off, dsc.evicted, dsc.window);
    if (tok >= dsc.n_old) continue;  // a slot of this step's new tokens, or never written
    const int64_t rel = tok - dsc.rope_base;
    if (rel < 0 || rel >= v.t_rows) {
      record_error(v.status, DEV_BOUNDS, 4, static_cast<int>(rel));
      continue;
    }
    const float c = v.rope_table[(rel * half + i) * 2], s = v.rope_table[(rel * half + i) * 2 + 1];
    const int64_t o = base + static_cast<int64_t>(off) * d;
    const float xa = bf16_to_f32(v.k_raw[o + i]), xb = bf16_to_f32(v.k_raw[o + i + half]);
    v.k_rot[o + i] = f32_to_f16(xa * c - xb * s);
    v.k_rot[o + i + half] = f32_to_f16(xa * s + xb * c);
  }
}

}  // namespace

cudaError_t launch_append_rope(const DevView& v, int n_active, int layer, const uint16_t* k, const uint16_t* vv,
                               cudaStream_t st) {
  dim3 grid(n_active * v.q_per_step, (v.n_kv_heads + kWarps - 1) / kWarps);
  append_rope_kernel<<<grid, kWarps * 32, 0, st>>>(v, layer, k, vv);
  return cudaGetLastError();
}

cudaError_t launch_rebase(const DevView& v, int n_active, int layer, cudaStream_t st) {
  dim3 grid(n_active, v.max_pages, v.n_kv_heads);
  rebase_kernel<<<grid, 128, 0, st>>>(v, layer);
  return cudaGetLastError();
}

}  // namespace rkv

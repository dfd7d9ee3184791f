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
//
// Both kernels move 16-byte chunks: a thread owns chunk c (elements 8c ..
// 8c+7) and its rotation partner c + d/16 (elements + d/2) of one key row,
// written at their swizzled chunk positions (rkv_internal.cuh).
#include "rkv_internal.cuh"

namespace rkv {
namespace {

__device__ __forceinline__ void unpack8(const uint4 u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = __uint_as_float(w[j] << 16);
    x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_f16(lo)) | (static_cast<uint32_t>(f32_to_f16(hi)) << 16);
}

// Rotate 8 pairs: xa[j] with xb[j] by (cos, sin) cs[2j], cs[2j+1]; fp16 out.
__device__ __forceinline__ void rotate8(const float (&xa)[8], const float (&xb)[8], const float* cs, uint4* ya,
                                        uint4* yb, bool* fits) {
  float ra[8], rb[8];
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float c = cs[2 * j], s = cs[2 * j + 1];
    ra[j] = xa[j] * c - xb[j] * s;
    rb[j] = xa[j] * s + xb[j] * c;
    ok = ok && fits_f16(ra[j]) && fits_f16(rb[j]);
  }
  *ya = make_uint4(pack_h2(ra[0], ra[1]), pack_h2(ra[2], ra[3]), pack_h2(ra[4], ra[5]), pack_h2(ra[6], ra[7]));
  *yb = make_uint4(pack_h2(rb[0], rb[1]), pack_h2(rb[2], rb[3]), pack_h2(rb[4], rb[5]), pack_h2(rb[6], rb[7]));
  *fits = ok;
}

// One thread per (layer, active stream, new token, kv head, chunk pair).
__global__ void __launch_bounds__(128) append_rope_kernel(DevView v, int layer0, int n_rows, const uint16_t* __restrict__ k,
                                                          const uint16_t* __restrict__ val, int64_t kv_layer_stride) {
  pdl_wait();
  pdl_launch_dependents();
  const int d = v.head_dim, half = d / 2, cpairs = d / 16, hkv = v.n_kv_heads;
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t per_layer = static_cast<int64_t>(n_rows) * hkv * cpairs;
  const int lz = blockIdx.y;
  if (idx >= per_layer) return;
  const int cp = static_cast<int>(idx % cpairs);
  const int kvh = static_cast<int>((idx / cpairs) % hkv);
  const int row = static_cast<int>(idx / (static_cast<int64_t>(cpairs) * hkv));  // a * Q + t
  const int layer = layer0 + lz;
  const int a = row / v.q_per_step, t = row % v.q_per_step;
  const StepDesc dsc = v.desc[a];
  const int64_t tok = dsc.n_old + t;
  const int slot = static_cast<int>(tok % dsc.ring);
  const int ring_page = slot / v.page_size;
  if (ring_page >= v.max_pages) {
    record_error(v.status, DEV_BOUNDS, 1, ring_page);
    return;
  }
  const int page = v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + ring_page];
  if (page < 0 || page >= v.n_pages) {
    record_error(v.status, DEV_BOUNDS, 2, page);
    return;
  }
  const int off = slot % v.page_size;
  const int64_t dst = pool_offset(v, layer, page, kvh, off);
  const int pa = swizzle_chunk(cp, off) * 8, pb = swizzle_chunk(cp + cpairs, off) * 8;
  const int64_t src = lz * kv_layer_stride + (static_cast<int64_t>(row) * hkv + kvh) * d;
  const uint4 ka = *reinterpret_cast<const uint4*>(k + src + cp * 8);
  const uint4 kb = *reinterpret_cast<const uint4*>(k + src + half + cp * 8);
  *reinterpret_cast<uint4*>(v.v + dst + pa) = *reinterpret_cast<const uint4*>(val + src + cp * 8);
  *reinterpret_cast<uint4*>(v.v + dst + pb) = *reinterpret_cast<const uint4*>(val + src + half + cp * 8);
  if (v.k_raw) {
    *reinterpret_cast<uint4*>(v.k_raw + dst + pa) = ka;
    *reinterpret_cast<uint4*>(v.k_raw + dst + pb) = kb;
  }
  float xa[8], xb[8];
  unpack8(ka, xa);
  unpack8(kb, xb);
  const float* cs = v.cs_new + (static_cast<int64_t>(row) * half + cp * 8) * 2;
  uint4 ya, yb;
  bool fits;
  rotate8(xa, xb, cs, &ya, &yb, &fits);
  if (!fits) record_error(v.status, DEV_RANGE, 1, cp);
  *reinterpret_cast<uint4*>(v.k_rot + dst + pa) = ya;
  *reinterpret_cast<uint4*>(v.k_rot + dst + pb) = yb;
}

// The fp8 store (kv_format e4m3): the same threads (one per chunk pair of a (row, kv head); the
// d/16 threads of a row are consecutive lanes), each rotating its 16 key elements in fp32 as above
// but with every product and sum rounded on its own, so that the code each element rounds to is a
// function of fp32 arithmetic that a reference can repeat exactly;
// the row's largest magnitude, of the rotated key and of the value separately, comes from a
// butterfly over those lanes, fixes the row's scale 2^e, and each element is stored as the e4m3
// code of x / 2^e (bytes, unswizzled: element i at byte i of the row) with the scales beside.
// Threads past the last row take part in the butterfly with zeros and store nothing.
__global__ void __launch_bounds__(128) append_rope_e4m3_kernel(DevView v, int layer0, int n_rows,
                                                               const uint16_t* __restrict__ k,
                                                               const uint16_t* __restrict__ val, int64_t kv_layer_stride) {
  pdl_wait();
  pdl_launch_dependents();
  const int d = v.head_dim, half = d / 2, cpairs = d / 16, hkv = v.n_kv_heads;
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t per_layer = static_cast<int64_t>(n_rows) * hkv * cpairs;
  const int lz = blockIdx.y;
  bool live = idx < per_layer;
  const int64_t id = live ? idx : 0;
  const int cp = static_cast<int>(id % cpairs);
  const int kvh = static_cast<int>((id / cpairs) % hkv);
  const int row = static_cast<int>(id / (static_cast<int64_t>(cpairs) * hkv));  // a * Q + t
  const int layer = layer0 + lz;
  const int a = row / v.q_per_step, t = row % v.q_per_step;
  const StepDesc dsc = v.desc[a];
  const int slot = static_cast<int>((dsc.n_old + t) % dsc.ring);
  const int ring_page = slot / v.page_size;
  int page = -1;
  if (live && ring_page >= v.max_pages) {
    record_error(v.status, DEV_BOUNDS, 1, ring_page);
    live = false;
  }
  if (live) {
    page = v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + ring_page];
    if (page < 0 || page >= v.n_pages) {
      record_error(v.status, DEV_BOUNDS, 2, page);
      live = false;
    }
  }
  float ra[8], rb[8], va[8], vb[8];
  float km = 0.f, vm = 0.f;
  bool ok = true;
  const int64_t src = lz * kv_layer_stride + (static_cast<int64_t>(row) * hkv + kvh) * d;
  if (live) {
    float xa[8], xb[8];
    unpack8(*reinterpret_cast<const uint4*>(k + src + cp * 8), xa);
    unpack8(*reinterpret_cast<const uint4*>(k + src + half + cp * 8), xb);
    unpack8(*reinterpret_cast<const uint4*>(val + src + cp * 8), va);
    unpack8(*reinterpret_cast<const uint4*>(val + src + half + cp * 8), vb);
    const float* cs = v.cs_new + (static_cast<int64_t>(row) * half + cp * 8) * 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // each product and sum rounded to fp32 (no fused multiply-add)
      const float c = cs[2 * j], sn = cs[2 * j + 1];
      ra[j] = __fsub_rn(__fmul_rn(xa[j], c), __fmul_rn(xb[j], sn));
      rb[j] = __fadd_rn(__fmul_rn(xa[j], sn), __fmul_rn(xb[j], c));
      ok = ok && fits_f16(ra[j]) && fits_f16(rb[j]);
      km = fmaxf(km, fmaxf(fabsf(ra[j]), fabsf(rb[j])));
      vm = fmaxf(vm, fmaxf(fabsf(va[j]), fabsf(vb[j])));
    }
  }
  for (int o = 1; o < cpairs; o <<= 1) {
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
  }
  if (!live) return;
  if (!ok) record_error(v.status, DEV_RANGE, 1, cp);
  // values are read back as fp16 code * 2^e: a row must stay clear of the fp16 limit after rounding
  if (!(vm < 61440.f)) record_error(v.status, DEV_RANGE, 2, cp);
  const int ek = e4m3_row_exponent(km), ev = e4m3_row_exponent(vm);
  const int off = slot % v.page_size;
  const int64_t dst = pool_offset(v, layer, page, kvh, off);  // = row index * d: a byte offset here
  uint8_t* k8 = reinterpret_cast<uint8_t*>(v.k_rot);
  uint8_t* v8 = reinterpret_cast<uint8_t*>(v.v);
  *reinterpret_cast<uint2*>(k8 + dst + cp * 8) = quantize8(ra, exp2_int(-ek));
  *reinterpret_cast<uint2*>(k8 + dst + half + cp * 8) = quantize8(rb, exp2_int(-ek));
  *reinterpret_cast<uint2*>(v8 + dst + cp * 8) = quantize8(va, exp2_int(-ev));
  *reinterpret_cast<uint2*>(v8 + dst + half + cp * 8) = quantize8(vb, exp2_int(-ev));
  if (cp == 0) v.kv_scale[dst / d] = make_float2(exp2_int(ek), exp2_int(ev));
}

// A thread re-bases one chunk pair (elements 8c .. 8c+7 and their partners
// + d/2) of one kv head for a run of kRebaseRun consecutive ring slots of one
// stream and layer.  Consecutive slots hold consecutive window positions
// (except where the ring wraps), so the cos/sin of the next slot's angles
// follow from the current ones by one complex multiplication with
// (cos, sin)(omega_i); the table row is read only for the run's first slot
// and after a wrap (at most 8 multiplications: ~1e-6 relative, far below the
// fp16 rounding of the result).  All of the run's key loads are issued before
// any arithmetic.  For a stream that re-bases this step, every retained key
// written before the step (tokens evicted .. n_old - 1) becomes
// R(j - rope_base) applied to its pre-RoPE copy: the exact result of rotating
// the previously stored key by R(-delta), with one rounding however many
// re-bases the key has seen.
constexpr int kRebaseThreads = 128;
constexpr int kRebaseRun = 8;  // divides every page size (16 .. 128)

// Four blocks per SM (at most 128 registers a thread): more runs' loads in flight while other
// runs compute.
__global__ void __launch_bounds__(kRebaseThreads, 4) rebase_kernel(DevView v, int layer0) {
  pdl_wait();
  pdl_launch_dependents();
  const int d = v.head_dim, half = d / 2, cpairs = d / 16;
  const int a = blockIdx.y;
  // layers in reverse block order: the last keys re-based are layer 0's, which decode attention
  // (layer-major) reads first, while they are still in L2
  const int lz = static_cast<int>(gridDim.z) - 1 - static_cast<int>(blockIdx.z);
  const StepDesc dsc = v.desc[a];
  if (dsc.delta == 0) return;
  const int item = blockIdx.x * kRebaseThreads + threadIdx.x;
  const int cp = item % cpairs;
  const int kvh = (item / cpairs) % v.n_kv_heads;
  const int slot0 = (item / (cpairs * v.n_kv_heads)) * kRebaseRun;
  const int W = dsc.ring;  // the ring's modulus
  if (slot0 >= W) return;
  const int ev_mod = static_cast<int>(dsc.evicted % W);
  const int old_len = static_cast<int>(dsc.n_old - dsc.evicted);  // window index of the first new token
  const int rel_shift = static_cast<int>(dsc.evicted - dsc.rope_base);
  const int page = v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + slot0 / v.page_size];
  if (page < 0 || page >= v.n_pages) {
    record_error(v.status, DEV_BOUNDS, 3, page);
    return;
  }
  const int64_t row0 = pool_offset(v, layer0 + lz, page, kvh, slot0 % v.page_size);
  uint4 ka[kRebaseRun], kb[kRebaseRun];
  int rel[kRebaseRun];
  bool live[kRebaseRun];
#pragma unroll
  for (int j = 0; j < kRebaseRun; ++j) {
    const int slot = slot0 + j;
    int w = slot - ev_mod;  // window index of the slot's token
    if (w < 0) w += W;
    live[j] = slot < W && w < old_len;  // retained tokens from before this step
    rel[j] = w + rel_shift;
    if (live[j] && (rel[j] < 0 || rel[j] >= v.t_rows)) {
      record_error(v.status, DEV_BOUNDS, 4, rel[j]);
      live[j] = false;
    }
    if (live[j]) {
      const int off = (slot0 + j) % v.page_size;
      const int64_t o = row0 + static_cast<int64_t>(j) * d;
      ka[j] = *reinterpret_cast<const uint4*>(v.k_raw + o + swizzle_chunk(cp, off) * 8);
      kb[j] = *reinterpret_cast<const uint4*>(v.k_raw + o + swizzle_chunk(cp + cpairs, off) * 8);
    }
  }
  // (cos, sin)(omega_i) of this thread's eight frequencies: table row 1
  // Coefficients in packed pairs of adjacent frequencies (i, i+1): c2[p] = (cos, cos), s2[p] =
  // (sin, sin) of frequencies 8cp + 2p, 8cp + 2p + 1; the rotation and the recurrence run on
  // paired fp32 FMAs (each lane rounds exactly as a scalar FMA).
  float2 c1[4], s1[4], ns1[4], c2[4], s2[4];
  if (v.t_rows > 1) {  // (cos, sin)(omega_i): table row 1 (a window of one key keeps nothing to re-base)
    const float4* t1 = reinterpret_cast<const float4*>(v.rope_table + (static_cast<int64_t>(1) * half + cp * 8) * 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 t = t1[q];
      c1[q] = make_float2(t.x, t.z);
      s1[q] = make_float2(t.y, t.w);
      ns1[q] = make_float2(-t.y, -t.w);
    }
  }
  int rel_cur = -2;
#pragma unroll
  for (int j = 0; j < kRebaseRun; ++j) {
    if (!live[j]) continue;
    if (rel[j] == rel_cur + 1) {  // advance by one position: (c, s) <- (c, s) * (cos, sin)(omega)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 c = c2[q], sn = s2[q];
        c2[q] = __ffma2_rn(c, c1[q], __fmul2_rn(sn, ns1[q]));
        s2[q] = __ffma2_rn(sn, c1[q], __fmul2_rn(c, s1[q]));
      }
    } else {  // first live slot of the run, or the ring wrapped: read the row
      const float4* t4 = reinterpret_cast<const float4*>(v.rope_table + (static_cast<int64_t>(rel[j]) * half + cp * 8) * 2);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 t = t4[q];
        c2[q] = make_float2(t.x, t.z);
        s2[q] = make_float2(t.y, t.w);
      }
    }
    rel_cur = rel[j];
    // (a, b) -> (a cos - b sin, a sin + b cos) on pairs of adjacent elements
    const uint32_t wa[4] = {ka[j].x, ka[j].y, ka[j].z, ka[j].w}, wb[4] = {kb[j].x, kb[j].y, kb[j].z, kb[j].w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 xa = make_float2(__uint_as_float(wa[q] << 16), __uint_as_float(wa[q] & 0xFFFF0000u));
      const float2 nxb = make_float2(-__uint_as_float(wb[q] << 16), -__uint_as_float(wb[q] & 0xFFFF0000u));
      const float2 xb = make_float2(-nxb.x, -nxb.y);
      const float2 ra = __ffma2_rn(nxb, s2[q], __fmul2_rn(xa, c2[q]));
      const float2 rb = __ffma2_rn(xa, s2[q], __fmul2_rn(xb, c2[q]));
      const __half2 ha = __floats2half2_rn(ra.x, ra.y), hb = __floats2half2_rn(rb.x, rb.y);
      ya[q] = *reinterpret_cast<const uint32_t*>(&ha);
      yb[q] = *reinterpret_cast<const uint32_t*>(&hb);
    }
    const int off = (slot0 + j) % v.page_size;
    const int64_t o = row0 + static_cast<int64_t>(j) * d;
    *reinterpret_cast<uint4*>(v.k_rot + o + swizzle_chunk(cp, off) * 8) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    *reinterpret_cast<uint4*>(v.k_rot + o + swizzle_chunk(cp + cpairs, off) * 8) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
  }
}

}  // namespace

cudaError_t launch_append_rope(const DevView& v, int n_active, int layer0, int n_layers, const uint16_t* k,
                               const uint16_t* vv, int64_t kv_layer_stride, cudaStream_t st) {
  const int n_rows = n_active * v.q_per_step;
  const int64_t per_layer = static_cast<int64_t>(n_rows) * v.n_kv_heads * (v.head_dim / 16);
  dim3 grid(static_cast<unsigned>((per_layer + 127) / 128), n_layers);
  if (v.kv_scale)
    return launch_pdl(append_rope_e4m3_kernel, grid, dim3(128), 0, st, v, layer0, n_rows, k, vv, kv_layer_stride);
  return launch_pdl(append_rope_kernel, grid, dim3(128), 0, st, v, layer0, n_rows, k, vv, kv_layer_stride);
}

cudaError_t launch_rebase(const DevView& v, int n_active, int layer0, int n_layers, cudaStream_t st) {
  if (v.scheme != RKV_SCHEME_EXACT_REBASE) return cudaSuccess;  // on read: nothing is stored re-based
  const int64_t per_stream =
      static_cast<int64_t>(v.max_pages) * v.page_size / kRebaseRun * v.n_kv_heads * (v.head_dim / 16);
  dim3 grid(static_cast<unsigned>((per_stream + kRebaseThreads - 1) / kRebaseThreads), n_active, n_layers);
  return launch_pdl(rebase_kernel, grid, dim3(kRebaseThreads), 0, st, v, layer0);
}

}  // namespace rkv

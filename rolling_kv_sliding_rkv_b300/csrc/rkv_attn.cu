// Windowed GQA attention over the ring (Audio8 ASR Infinite 无限长转写原理,
// "Rolling KV Cache 三步拆解", 第 3 步: attention scans only the fixed window,
// so the cost of a step is constant), split over the window's pages, then a
// log-sum-exp merge of the splits.
//
// Split (stream a, kv head, split c) covers ring slots
// [c * pages_per_split * page_size, ...) of stream a.  Slot order is not
// token order, which softmax does not care about; a slot whose token is not
// in [evicted, n_new) is empty.  Query token n_old + t attends key token j iff
// j <= n_old + t (causal inside a multi-query step; every stored token is in
// the window by construction of the ring).
//
// The step's queries arrive pre-RoPE (bf16) and are rotated here, in fp32,
// with the cos/sin of their positions computed once per step; they are never
// rounded back to a 16-bit format.  Keys are read as the stored fp16 rotated
// keys, values as bf16.
//
// Partial results per (a, query row, split): m = max scaled score in log2
// units, l = sum 2^(s - m), o = sum 2^(s - m) v / l.
#include <math_constants.h>

#include "rkv_internal.cuh"

namespace rkv {
namespace {

constexpr int kWarps = 4;

template <int D, int R>
__global__ void __launch_bounds__(kWarps * 32) attn_partial_kernel(DevView v, int layer,
                                                                   const uint16_t* __restrict__ q) {
  constexpr int E = D / 32;  // elements of a head vector per lane
  const int splits = v.splits;
  const int a = blockIdx.x / splits, c = blockIdx.x % splits, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = v.n_q_heads, group = hq / v.n_kv_heads, nq = v.q_per_step;
  const int rows = group * nq;
  const StepDesc dsc = v.desc[a];

  __shared__ float qs[R][D];
  __shared__ float red_ml[kWarps][R][2];
  __shared__ float red_o[kWarps][R][D];

  constexpr int H = D / 2;
  for (int e = threadIdx.x; e < R * H; e += blockDim.x) {
    const int r = e / H, i = e % H;
    float ya = 0.f, yb = 0.f;
    if (r < rows) {
      const int t = r / group, h = kvh * group + r % group;
      const uint16_t* x = q + ((static_cast<int64_t>(a) * nq + t) * hq + h) * D;
      const float* cs = v.cs_new + ((static_cast<int64_t>(a) * nq + t) * H + i) * 2;
      const float xa = bf16_to_f32(x[i]), xb = bf16_to_f32(x[i + H]);
      ya = xa * cs[0] - xb * cs[1];
      yb = xa * cs[1] + xb * cs[0];
    }
    qs[r][i] = ya;
    qs[r][i + H] = yb;
  }
  __syncthreads();

  float qreg[R][E], acc[R][E], m[R], l[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -CUDART_INF_F;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      qreg[r][e] = qs[r][lane * E + e];
      acc[r][e] = 0.f;
    }
  }

  const int64_t n_new = dsc.n_old + nq;
  const int span = v.pages_per_split * v.page_size;
  const int s0 = c * span;
  const int s1 = min(s0 + span, dsc.window);
  for (int slot = s0 + warp; slot < s1; slot += kWarps) {
    const int64_t tok = token_in_slot(slot, dsc.evicted, dsc.window);
    if (tok >= n_new) continue;
    const int page = v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + slot / v.page_size];
    if (page < 0 || page >= v.n_pages) {
      if (lane == 0) record_error(v.status, DEV_BOUNDS, 5, page);
      continue;
    }
    const int64_t off = pool_offset(v, layer, page, kvh, slot % v.page_size) + lane * E;
    float kf[E], vf[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kf[e] = f16_to_f32(v.k_rot[off + e]);
      vf[e] = bf16_to_f32(v.v[off + e]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r >= rows) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(qreg[r][e], kf[e], dot);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (tok > dsc.n_old + r / group) continue;  // causal inside the step
      const float s2 = dot * v.scale_log2;
      const float m_new = fmaxf(m[r], s2);
      const float alpha = exp2f(m[r] - m_new);
      const float p = exp2f(s2 - m_new);
      l[r] = l[r] * alpha + p;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] = fmaf(acc[r][e], alpha, p * vf[e]);
      m[r] = m_new;
    }
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (lane == 0) {
      red_ml[warp][r][0] = m[r];
      red_ml[warp][r][1] = l[r];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) red_o[warp][r][lane * E + e] = acc[r][e];
  }
  __syncthreads();

  const int qhq = nq * hq;
  for (int e = threadIdx.x; e < rows * D; e += blockDim.x) {
    const int r = e / D, i = e % D;
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red_ml[w][r][0]);
    float lsum = 0.f, osum = 0.f;
    if (mx != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(red_ml[w][r][0] - mx);
        lsum += red_ml[w][r][1] * f;
        osum += red_o[w][r][i] * f;
      }
    }
    const int t = r / group, h = kvh * group + r % group;
    const int64_t prow = (static_cast<int64_t>(a) * qhq + t * hq + h) * splits + c;
    v.part_o[prow * D + i] = lsum > 0.f ? osum / lsum : 0.f;
    if (i == 0) {
      v.part_ml[prow * 2] = mx;
      v.part_ml[prow * 2 + 1] = lsum;
    }
  }
}

// One block per (active stream, query row): combine the splits.
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(DevView v, uint16_t* __restrict__ out, float* __restrict__ lse) {
  const int splits = v.splits;
  const int64_t prow0 = static_cast<int64_t>(blockIdx.x) * splits;
  const float* ml = v.part_ml + prow0 * 2;
  float mx = -CUDART_INF_F;
  for (int c = 0; c < splits; ++c)
    if (ml[2 * c + 1] > 0.f) mx = fmaxf(mx, ml[2 * c]);
  float lsum = 0.f;
  for (int c = 0; c < splits; ++c)
    if (ml[2 * c + 1] > 0.f) lsum += ml[2 * c + 1] * exp2f(ml[2 * c] - mx);
  for (int i = threadIdx.x; i < D; i += blockDim.x) {
    float o = 0.f;
    for (int c = 0; c < splits; ++c)
      if (ml[2 * c + 1] > 0.f) o += ml[2 * c + 1] * exp2f(ml[2 * c] - mx) * v.part_o[(prow0 + c) * D + i];
    out[static_cast<int64_t>(blockIdx.x) * D + i] = f32_to_bf16(o / lsum);
  }
  if (lse && threadIdx.x == 0) lse[blockIdx.x] = (mx + log2f(lsum)) * 0.69314718055994531f;
}

template <int D, int R>
cudaError_t launch_partial(const DevView& v, int n_active, int layer, const uint16_t* q, cudaStream_t st) {
  dim3 grid(n_active * v.splits, v.n_kv_heads);
  attn_partial_kernel<D, R><<<grid, kWarps * 32, 0, st>>>(v, layer, q);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_partial_d(const DevView& v, int n_active, int layer, const uint16_t* q, cudaStream_t st) {
  const int rows = v.n_q_heads / v.n_kv_heads * v.q_per_step;
  if (rows <= 1) return launch_partial<D, 1>(v, n_active, layer, q, st);
  if (rows <= 2) return launch_partial<D, 2>(v, n_active, layer, q, st);
  if (rows <= 4) return launch_partial<D, 4>(v, n_active, layer, q, st);
  if (rows <= 8) return launch_partial<D, 8>(v, n_active, layer, q, st);
  return launch_partial<D, 16>(v, n_active, layer, q, st);
}

}  // namespace

cudaError_t launch_decode_attn(const DevView& v, int n_active, int layer, const uint16_t* q, uint16_t* out,
                               float* lse, cudaStream_t st) {
  cudaError_t err;
  const int blocks = n_active * v.q_per_step * v.n_q_heads;
  if (v.head_dim == 128) {
    err = launch_partial_d<128>(v, n_active, layer, q, st);
    if (err != cudaSuccess) return err;
    merge_kernel<128><<<blocks, 128, 0, st>>>(v, out, lse);
  } else {
    err = launch_partial_d<64>(v, n_active, layer, q, st);
    if (err != cudaSuccess) return err;
    merge_kernel<64><<<blocks, 64, 0, st>>>(v, out, lse);
  }
  return cudaGetLastError();
}

}  // namespace rkv

// RoPE angle tables and the begin-step kernel.
//
// Positions reach 10^6 (24 h at 12.5 Hz) and beyond; the explainer's "no
// drift in 24/7 runs" (Audio8 ASR Infinite 无限长转写原理, "Rolling KV Cache
// 三步拆解", 第 2 步) needs angles p * omega_i that do not lose precision with
// p, so every angle goes through rope_cos_sin (fp64, error-free product and
// three-part 2*pi reduction) once per step per stream, shared by all layers.
#include "rkv_internal.cuh"

namespace rkv {
namespace {

__global__ void rope_cossin_kernel(const int64_t* __restrict__ pos, int n, int half, Omegas w,
                                   float* __restrict__ cs) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  const int row = idx / half, i = idx % half;
  float c, s;
  rope_cos_sin(pos[row], w.w[i], &c, &s);
  cs[2 * idx] = c;
  cs[2 * idx + 1] = s;
}

// rope_table[r][i] = (cos, sin)(r * omega_i) for the window-relative positions
// of the exact scheme, r < t_rows.
__global__ void init_tables_kernel(DevView v) {
  const int half = v.head_dim / 2;
  const int64_t total = static_cast<int64_t>(v.t_rows) * half;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx / half;
    const int i = static_cast<int>(idx % half);
    float c, s;
    rope_cos_sin(r, v.omega[i], &c, &s);
    v.rope_table[2 * idx] = c;
    v.rope_table[2 * idx + 1] = s;
  }
}

// One block per active stream: advance the ring state (host-side rules in
// rkv.h, rkv_begin_step), record the step descriptor, then cos/sin of the
// positions of the step's new tokens.
__global__ void begin_step_kernel(DevView v, ActiveIds ids) {
  pdl_wait();
  pdl_launch_dependents();
  const int a = blockIdx.x;
  const int s = ids.id[a];
  __shared__ int64_t pos0;
  if (threadIdx.x == 0) {
    int64_t* st = v.state + static_cast<int64_t>(s) * kStateFields;
    const int64_t n_old = st[F_N];
    const int64_t w = st[F_W];
    const int64_t p0 = st[F_P0];
    int64_t rope_base = st[F_ROPE_BASE];
    const int64_t n = n_old + v.q_per_step;
    const int64_t len = n < w ? n : w;
    const int64_t ev = n - len;
    int64_t delta = 0;
    if (exact_scheme(v.scheme) && ev - rope_base >= v.rebase_interval) {
      delta = ev - rope_base;
      rope_base = ev;
    }
    st[F_N] = n;
    st[F_LEN] = len;
    st[F_EVICTED] = ev;
    st[F_KV_POS_OFFSET] = p0 + ev;
    st[F_ROPE_BASE] = rope_base;
    st[F_HEAD_SLOT] = ev % w;
    StepDesc d;
    d.n_old = n_old;
    d.evicted = ev;
    d.rope_base = rope_base;
    d.delta = delta;
    d.stream = s;
    d.len = static_cast<int32_t>(len);
    d.window = static_cast<int32_t>(w);
    d.pad = 0;
    v.desc[a] = d;
    // the logical position P0 + j (offset-only), or j - rope_base (exact)
    pos0 = exact_scheme(v.scheme) ? n_old - rope_base : p0 + n_old;
  }
  __syncthreads();
  const int half = v.head_dim / 2;
  for (int idx = threadIdx.x; idx < v.q_per_step * half; idx += blockDim.x) {
    const int t = idx / half, i = idx % half;
    float c, sn;
    rope_cos_sin(pos0 + t, v.omega[i], &c, &sn);
    float* dst = v.cs_new + ((static_cast<int64_t>(a) * v.q_per_step + t) * half + i) * 2;
    dst[0] = c;
    dst[1] = sn;
  }
}

// One thread: empty stream s (its pages keep stale data, which the ring
// bookkeeping masks: slots at or beyond len are never read before rewritten).
__global__ void reset_stream_kernel(DevView v, int s, int64_t p0) {
  int64_t* st = v.state + static_cast<int64_t>(s) * kStateFields;
  st[F_N] = 0;
  st[F_LEN] = 0;
  st[F_EVICTED] = 0;
  st[F_KV_POS_OFFSET] = p0;
  st[F_ROPE_BASE] = 0;
  st[F_HEAD_SLOT] = 0;
  st[F_P0] = p0;  // F_W is kept: the stream's pages fix its window
}

}  // namespace

cudaError_t launch_reset_stream(const DevView& v, int s, int64_t p0, cudaStream_t st) {
  reset_stream_kernel<<<1, 1, 0, st>>>(v, s, p0);
  return cudaGetLastError();
}

cudaError_t launch_rope_cossin(const int64_t* pos, int n, int head_dim, const Omegas& w, float* cs,
                               cudaStream_t st) {
  const int half = head_dim / 2;
  const int total = n * half;
  if (total == 0) return cudaSuccess;
  rope_cossin_kernel<<<(total + 255) / 256, 256, 0, st>>>(pos, n, half, w, cs);
  return cudaGetLastError();
}

cudaError_t launch_init_tables(const DevView& v, cudaStream_t st) {
  if (v.t_rows > 0) {
    const int64_t total = static_cast<int64_t>(v.t_rows) * (v.head_dim / 2);
    const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    init_tables_kernel<<<blocks, 256, 0, st>>>(v);
  }
  return cudaGetLastError();
}

cudaError_t launch_begin_step(const DevView& v, const ActiveIds& ids, cudaStream_t st) {
  return launch_pdl(begin_step_kernel, dim3(ids.n), dim3(64), 0, st, v, ids);
}

}  // namespace rkv

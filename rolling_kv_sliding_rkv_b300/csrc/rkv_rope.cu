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
//
// Positions per scheme, for new token j = n_old + t:
//   offset-only         keys and queries at P0 + j;
//   exact re-base       keys and queries at j - rope_base (window-relative);
//   exact, on read      key stored at its ring slot j mod C (C = W +
//                       window_slack, the ring's capacity); the query at
//                       j - C * floor(evicted / C) against the keys of ring
//                       slots >= evicted mod C, and C less against the slots
//                       below (tokens of the ring's next lap), the second by
//                       the rotation R(-C) the kernel applies to the first.
//   Every score then sees the position difference of its two tokens.
__global__ void begin_step_kernel(DevView v, ActiveIds ids) {
  pdl_wait();
  pdl_launch_dependents();
  const int a = blockIdx.x;
  const int s = ids.id[a];
  __shared__ int64_t pos0, qpos0, win;
  if (threadIdx.x == 0) {
    int64_t* st = v.state + static_cast<int64_t>(s) * kStateFields;
    const int64_t n_old = st[F_N];
    const int64_t w = st[F_W];
    const int64_t p0 = st[F_P0];
    int64_t rope_base = st[F_ROPE_BASE];
    const int64_t ring = w + v.window_slack;  // ring capacity C
    const int64_t n = n_old + v.q_per_step;
    // keep every token while they fit in the ring; when this step's would not, evict down to the
    // last W in one batch (window_slack = 0: exactly enough every step, a plain sliding window)
    const int64_t ev = n - st[F_EVICTED] > ring ? n - w : st[F_EVICTED];
    const int64_t len = n - ev;
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
    st[F_HEAD_SLOT] = ev % ring;
    StepDesc d;
    d.n_old = n_old;
    d.evicted = ev;
    d.rope_base = rope_base;
    d.delta = delta;
    d.stream = s;
    d.len = static_cast<int32_t>(len);
    d.ring = static_cast<int32_t>(ring);
    d.pad = 0;
    v.desc[a] = d;
    // the logical position P0 + j (offset-only), j - rope_base (exact re-base), or the ring lap's
    // origin for the queries of the on-read scheme (keys: their slot, below)
    pos0 = v.scheme == RKV_SCHEME_EXACT_REBASE ? n_old - rope_base : p0 + n_old;
    qpos0 = n_old - (ev / ring) * ring;
    win = ring;
  }
  __syncthreads();
  const int half = v.head_dim / 2;
  const bool on_read = v.scheme == RKV_SCHEME_EXACT_ON_READ;
  for (int idx = threadIdx.x; idx < v.q_per_step * half; idx += blockDim.x) {
    const int t = idx / half, i = idx % half;
    const int64_t row = ((static_cast<int64_t>(a) * v.q_per_step + t) * half + i) * 2;
    float c, sn;
    rope_cos_sin(on_read ? (qpos0 + t) % win : pos0 + t, v.omega[i], &c, &sn);
    v.cs_new[row] = c;
    v.cs_new[row + 1] = sn;
    if (on_read) {
      rope_cos_sin(qpos0 + t, v.omega[i], &c, &sn);
      v.cs_q[row] = c;
      v.cs_q[row + 1] = sn;
    }
  }
  if (on_read)
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
      float c, sn;
      rope_cos_sin(-win, v.omega[i], &c, &sn);
      v.cs_lap[(static_cast<int64_t>(a) * half + i) * 2] = c;
      v.cs_lap[(static_cast<int64_t>(a) * half + i) * 2 + 1] = sn;
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

// One thread per entry of a device-side list: reset stream ids[i] to start offset p0[i] (as
// reset_stream_kernel); negative ids are skipped, entries out of range are reported.
__global__ void reset_streams_kernel(DevView v, const int32_t* __restrict__ ids, const int64_t* __restrict__ p0,
                                     int n) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int s = ids[i];
  const int64_t start = p0[i];
  if (s < 0) return;
  if (s >= v.n_streams || start < 0 || start >= (int64_t(1) << 52)) {
    record_error(v.status, DEV_BOUNDS, 5, s);
    return;
  }
  int64_t* st = v.state + static_cast<int64_t>(s) * kStateFields;
  st[F_N] = 0;
  st[F_LEN] = 0;
  st[F_EVICTED] = 0;
  st[F_KV_POS_OFFSET] = start;
  st[F_ROPE_BASE] = 0;
  st[F_HEAD_SLOT] = 0;
  st[F_P0] = start;
}

}  // namespace

cudaError_t launch_reset_streams(const DevView& v, const int32_t* ids, const int64_t* p0, int n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(reset_streams_kernel, dim3((n + 127) / 128), dim3(128), 0, st, v, ids, p0, n);
}

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

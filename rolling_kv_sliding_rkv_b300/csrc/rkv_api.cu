// Host side of the C ABI declared in include/rkv.h: validation, the layout of
// the caller-owned device buffers, the per-step call order, error reporting.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "rkv_internal.cuh"

namespace {
// An NVTX range around each call that enqueues work (rkv:<call>), so a profiler can
// select one step or one call (ncu --nvtx --nvtx-include); free without a tool attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace

struct rkv_handle {
  rkv_config cfg;
  rkv::DevView view;
  size_t pool_bytes = 0, state_bytes = 0;
  int32_t w_max = 0;
  int device = 0;
  int num_sms = 0;
  bool step_open = false;
  bool launched_since_begin = false;  // a kernel of this library followed the begin-step kernel
  int32_t n_active = 0;
  std::vector<uint8_t> appended, rebased;
  std::vector<int32_t> first_page, n_pages_of;  // per stream: its contiguous run of pages
  int32_t regions = 0;           // planes of the pool: K, V (, pre-RoPE K | row scales)
  char* pool = nullptr;
  size_t region_elems = 0;       // elements (rows x d) of one plane
  std::string last_error;
};

namespace {

thread_local std::string g_last_error;

int fail(rkv_handle* h, int code, const std::string& msg) {
  (h ? h->last_error : g_last_error) = msg;
  return code;
}

int cuda_fail(rkv_handle* h, cudaError_t e, const char* what) {
  return fail(h, RKV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
  size_t state, page_table, desc, cs_new, cs_q, cs_lap, omega, rope_table, status, total;
  size_t pool_region_elems;  // elements (rows x d) of one pool plane (all layers)
  size_t pool_bytes;
  int32_t max_pages, n_pages, t_rows, w_max, regions;
};

bool validate_config(const rkv_config* c, std::string* why) {
  char buf[256];
  auto bad = [&](const char* m) { *why = m; return false; };
  if (!c) return bad("config is NULL");
  if (c->n_layers < 1 || c->n_layers > 4096) return bad("n_layers must be in [1, 4096]");
  if (c->n_streams < 1 || c->n_streams > RKV_MAX_STREAMS) return bad("n_streams must be in [1, RKV_MAX_STREAMS]");
  if (c->n_kv_heads < 1 || c->n_q_heads < 1 || c->n_q_heads % c->n_kv_heads != 0)
    return bad("n_q_heads must be a positive multiple of n_kv_heads");
  if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c->q_per_step < 1 || c->q_per_step > 8) return bad("q_per_step must be in [1, 8]");
  if (c->n_q_heads / c->n_kv_heads * c->q_per_step > 16) return bad("(n_q_heads / n_kv_heads) * q_per_step must be <= 16");
  if (c->n_q_heads > 256 || c->n_kv_heads > 256) return bad("at most 256 heads");
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64 && c->page_size != 128)
    return bad("page_size must be 16, 32, 64 or 128");
  if (c->scheme != RKV_SCHEME_OFFSET_ONLY && !rkv::exact_scheme(c->scheme)) return bad("unknown scheme");
  if (c->rebase_interval < 1) return bad("rebase_interval must be >= 1");
  if (c->window_slack < 0 || c->window_slack > RKV_MAX_WINDOW) return bad("window_slack must be in [0, RKV_MAX_WINDOW]");
  if (c->kv_format != RKV_KV_F16 && c->kv_format != RKV_KV_E4M3) return bad("unknown kv_format");
  if (c->reserved != 0) return bad("reserved must be 0");
  if (c->kv_format == RKV_KV_E4M3 && c->scheme == RKV_SCHEME_EXACT_REBASE)
    return bad("the fp8 store takes offset-only or the re-base applied on read, not the materialised re-base");
  if (c->kv_format == RKV_KV_E4M3 && c->n_q_heads / c->n_kv_heads * c->q_per_step > 8)
    return bad("the fp8 store needs (n_q_heads / n_kv_heads) * q_per_step <= 8");
  if (!(c->rope_theta > 1.0) || !std::isfinite(c->rope_theta)) return bad("rope_theta must be finite and > 1");
  if (!(c->softmax_scale >= 0.0) || !std::isfinite(c->softmax_scale)) return bad("softmax_scale must be finite and >= 0");
  (void)buf;
  return true;
}

bool compute_layout(const rkv_config* c, const int32_t* window, Layout* L, std::string* why) {
  if (!validate_config(c, why)) return false;
  if (!window) {
    *why = "window is NULL";
    return false;
  }
  const int S = c->n_streams;
  int32_t w_max = 0;
  int64_t n_pages = 0;
  for (int s = 0; s < S; ++s) {
    const int32_t w = window[s];
    if (w < c->q_per_step || w > RKV_MAX_WINDOW - c->window_slack) {
      char buf[160];
      snprintf(buf, sizeof buf, "window[%d] = %d outside [q_per_step, RKV_MAX_WINDOW - window_slack]", s, w);
      *why = buf;
      return false;
    }
    const int32_t ring = w + c->window_slack;  // the stream's ring capacity
    w_max = ring > w_max ? ring : w_max;
    n_pages += (ring + c->page_size - 1) / c->page_size;
  }
  if (n_pages > (1 << 30)) {
    *why = "too many pages";
    return false;
  }
  L->w_max = w_max;
  L->max_pages = (w_max + c->page_size - 1) / c->page_size;
  L->n_pages = static_cast<int32_t>(n_pages);
  const bool on_read = c->scheme == RKV_SCHEME_EXACT_ON_READ;
  // window-relative positions of the materialised exact re-base stay below C + interval - 1
  const int64_t t_rows =
      c->scheme == RKV_SCHEME_EXACT_REBASE ? static_cast<int64_t>(w_max) + c->rebase_interval - 1 : 0;
  if (t_rows > (1 << 24)) {
    *why = "window + rebase_interval too large";
    return false;
  }
  L->t_rows = static_cast<int32_t>(t_rows);
  // rotated keys, values, and pre-RoPE keys for the materialised exact re-base
  L->regions = c->scheme == RKV_SCHEME_EXACT_REBASE ? 3 : 2;
  const int half = c->head_dim / 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L->state = take(static_cast<size_t>(S) * rkv::kStateFields * sizeof(int64_t));
  L->page_table = take(static_cast<size_t>(S) * L->max_pages * sizeof(int32_t));
  L->desc = take(static_cast<size_t>(S) * sizeof(rkv::StepDesc));
  L->cs_new = take(static_cast<size_t>(S) * c->q_per_step * half * 2 * sizeof(float));
  L->cs_q = on_read ? take(static_cast<size_t>(S) * c->q_per_step * half * 2 * sizeof(float)) : L->cs_new;
  L->cs_lap = on_read ? take(static_cast<size_t>(S) * half * 2 * sizeof(float)) : 0;
  L->omega = take(static_cast<size_t>(half) * sizeof(double));
  L->rope_table = take(static_cast<size_t>(t_rows) * half * 2 * sizeof(float));
  L->status = take(4 * sizeof(int32_t));
  L->total = off;
  L->pool_region_elems = static_cast<size_t>(c->n_layers) * n_pages * c->n_kv_heads * c->page_size * c->head_dim;
  if (c->kv_format == RKV_KV_E4M3) {
    // planes: fp8 keys, fp8 values (one byte per element), and a (key, value) scale pair per row
    L->regions = 3;
    L->pool_bytes = 2 * L->pool_region_elems + L->pool_region_elems / c->head_dim * 2 * sizeof(float);
  } else {
    L->pool_bytes = L->pool_region_elems * L->regions * sizeof(uint16_t);
  }
  return true;
}

bool step_in_progress(const rkv_handle* h) {
  if (!h->step_open) return false;
  const bool exact = rkv::exact_scheme(h->cfg.scheme);
  for (int l = 0; l < h->cfg.n_layers; ++l)
    if (!h->appended[l] || (exact && !h->rebased[l])) return true;
  return false;
}

bool check_layer(rkv_handle* h, int32_t layer) { return layer >= 0 && layer < h->cfg.n_layers; }

// What the next decode-attention launch may read before its dependency wait: the begin-step
// kernel's outputs once another kernel of this library followed it (it is then two or more
// launches back), and the caller's queries only when they were written before the call
// (rkv_step) and the descriptors may be read as well.
int early_bits(const rkv_handle* h, bool q_before_call) {
  if (!h->launched_since_begin) return 0;
  return rkv::kEarlyDesc | (q_before_call ? rkv::kEarlyQ : 0);
}

}  // namespace

extern "C" {

int rkv_clock_resolve(int32_t frame_len, int32_t target_delay_ms, rkv_clock* out) {
  if (!out) return fail(nullptr, RKV_ERR_INVALID_ARG, "out is NULL");
  int left_pad;
  switch (frame_len) {  // Edge0/Audio8-ASR-Infinite README, "Optimized operation points"
    case 4: left_pad = 18; break;
    case 6: left_pad = 12; break;
    case 8: left_pad = 9; break;
    default: return fail(nullptr, RKV_ERR_CONFIG, "frame_len must be 4, 6 or 8");
  }
  const int32_t clock = 20 * frame_len;  // 20 ms tower frame (explainer, "三档音频时钟")
  if (target_delay_ms <= 0 || target_delay_ms % clock != 0)
    return fail(nullptr, RKV_ERR_CONFIG, "target_delay_ms must be a positive multiple of the clock");
  static const int32_t trained[3][4] = {{240, 320, 480, 560}, {240, 480, 0, 0}, {320, 480, 0, 0}};
  const int row = frame_len == 4 ? 0 : frame_len == 6 ? 1 : 2;
  int post = 0;
  for (int i = 0; i < 4; ++i) post |= trained[row][i] == target_delay_ms;
  out->clock_ms = clock;
  out->window = (30000 + clock - 1) / clock;  // 30 s native context, rounded up
  out->num_delay_tokens = target_delay_ms / clock;
  out->left_pad_tokens = left_pad;
  out->samples_per_token = 16000 * clock / 1000;
  out->post_trained = post;
  out->decisions_per_s = 1000.0 / clock;
  return RKV_OK;
}

int rkv_required_bytes(const rkv_config* cfg, const int32_t* window, size_t* pool_bytes, size_t* state_bytes) {
  if (!pool_bytes || !state_bytes) return fail(nullptr, RKV_ERR_INVALID_ARG, "size outputs are NULL");
  Layout L;
  std::string why;
  if (!compute_layout(cfg, window, &L, &why)) return fail(nullptr, cfg && window ? RKV_ERR_CONFIG : RKV_ERR_INVALID_ARG, why);
  *pool_bytes = L.pool_bytes;
  *state_bytes = L.total;
  return RKV_OK;
}

int rkv_create(const rkv_config* cfg, const int32_t* window, const int64_t* start_offset, void* pool_dev,
               size_t pool_bytes, void* state_dev, size_t state_bytes, void* stream, rkv_handle** out) {
  if (!out) return fail(nullptr, RKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  Layout L;
  std::string why;
  if (!cfg || !window || !start_offset) return fail(nullptr, RKV_ERR_INVALID_ARG, "config, window or start_offset is NULL");
  if (!compute_layout(cfg, window, &L, &why)) return fail(nullptr, RKV_ERR_CONFIG, why);
  for (int s = 0; s < cfg->n_streams; ++s)
    if (start_offset[s] < 0 || start_offset[s] >= (int64_t(1) << 52))
      return fail(nullptr, RKV_ERR_CONFIG, "start_offset must be in [0, 2^52)");
  if (!pool_dev || !state_dev) return fail(nullptr, RKV_ERR_INVALID_ARG, "pool_dev or state_dev is NULL");
  if ((reinterpret_cast<uintptr_t>(pool_dev) | reinterpret_cast<uintptr_t>(state_dev)) & (kAlign - 1))
    return fail(nullptr, RKV_ERR_INVALID_ARG, "device buffers must be 256-byte aligned");
  const size_t need_pool = L.pool_bytes;
  if (pool_bytes < need_pool || state_bytes < L.total)
    return fail(nullptr, RKV_ERR_CAPACITY, "pool or state buffer smaller than rkv_required_bytes");

  rkv_handle* h = new rkv_handle();
  h->cfg = *cfg;
  h->pool_bytes = pool_bytes;
  h->state_bytes = state_bytes;
  h->w_max = L.w_max;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(nullptr, e, "querying the device");
  }

  char* sb = static_cast<char*>(state_dev);
  rkv::DevView& v = h->view;
  v.state = reinterpret_cast<int64_t*>(sb + L.state);
  v.page_table = reinterpret_cast<int32_t*>(sb + L.page_table);
  v.desc = reinterpret_cast<rkv::StepDesc*>(sb + L.desc);
  v.cs_new = reinterpret_cast<float*>(sb + L.cs_new);
  v.cs_q = reinterpret_cast<float*>(sb + L.cs_q);
  v.cs_lap = cfg->scheme == RKV_SCHEME_EXACT_ON_READ ? reinterpret_cast<float*>(sb + L.cs_lap) : nullptr;
  v.omega = reinterpret_cast<double*>(sb + L.omega);
  v.rope_table = L.t_rows ? reinterpret_cast<float*>(sb + L.rope_table) : nullptr;
  v.part_ml = nullptr;  // split-K partials: only the scratch form of decode attention has them
  v.part_o = nullptr;
  v.status = reinterpret_cast<int32_t*>(sb + L.status);
  char* pool = static_cast<char*>(pool_dev);
  const bool kv8 = cfg->kv_format == RKV_KV_E4M3;
  const size_t plane_bytes = L.pool_region_elems * (kv8 ? 1 : sizeof(uint16_t));
  v.k_rot = reinterpret_cast<uint16_t*>(pool);  // fp8: the same plane read as bytes
  v.v = reinterpret_cast<uint16_t*>(pool + plane_bytes);
  v.k_raw = !kv8 && L.regions == 3 ? reinterpret_cast<uint16_t*>(pool + 2 * plane_bytes) : nullptr;
  v.kv_scale = kv8 ? reinterpret_cast<float2*>(pool + 2 * plane_bytes) : nullptr;
  v.layer_stride = static_cast<int64_t>(L.n_pages) * cfg->n_kv_heads * cfg->page_size * cfg->head_dim;
  v.n_streams = cfg->n_streams;
  v.n_layers = cfg->n_layers;
  v.n_q_heads = cfg->n_q_heads;
  v.n_kv_heads = cfg->n_kv_heads;
  v.head_dim = cfg->head_dim;
  v.q_per_step = cfg->q_per_step;
  v.page_size = cfg->page_size;
  v.n_pages = L.n_pages;
  v.max_pages = L.max_pages;
  v.t_rows = L.t_rows;
  v.scheme = cfg->scheme;
  v.rebase_interval = cfg->rebase_interval;
  v.window_slack = cfg->window_slack;
  const double scale = cfg->softmax_scale > 0.0 ? cfg->softmax_scale : 1.0 / std::sqrt(static_cast<double>(cfg->head_dim));
  v.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  v.num_sms = h->num_sms;
  v.wait_ns = rkv::kDefaultWaitNs;
  v.withhold_stage = -1;

  // host images of the stream state, page tables and RoPE frequencies
  const int S = cfg->n_streams, half = cfg->head_dim / 2;
  std::vector<int64_t> state(static_cast<size_t>(S) * rkv::kStateFields, 0);
  std::vector<int32_t> table(static_cast<size_t>(S) * L.max_pages, -1);
  int32_t next_page = 0;
  for (int s = 0; s < S; ++s) {
    int64_t* st = &state[static_cast<size_t>(s) * rkv::kStateFields];
    st[rkv::F_KV_POS_OFFSET] = start_offset[s];
    st[rkv::F_W] = window[s];
    st[rkv::F_P0] = start_offset[s];
    const int pages = (window[s] + cfg->window_slack + cfg->page_size - 1) / cfg->page_size;
    h->first_page.push_back(next_page);
    h->n_pages_of.push_back(pages);
    for (int p = 0; p < pages; ++p) table[static_cast<size_t>(s) * L.max_pages + p] = next_page++;
  }
  std::vector<double> omega(half);
  for (int i = 0; i < half; ++i) omega[i] = std::pow(cfg->rope_theta, -2.0 * i / cfg->head_dim);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // a zeroed pool keeps never-written slots finite (they are masked, but a masked
  // score still multiplies its value row by zero)
  e = cudaMemsetAsync(pool_dev, 0, need_pool, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(v.state, state.data(), state.size() * sizeof(int64_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(v.page_table, table.data(), table.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v.omega, omega.data(), half * sizeof(double), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.status, 0, 4 * sizeof(int32_t), st);
  if (e == cudaSuccess) e = rkv::launch_init_tables(v, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(nullptr, e, "initialising the device state");
  }
  h->appended.assign(cfg->n_layers, 0);
  h->rebased.assign(cfg->n_layers, 0);
  h->regions = L.regions;
  h->pool = pool;
  h->region_elems = L.pool_region_elems;
  *out = h;
  return RKV_OK;
}

int rkv_begin_step(rkv_handle* h, const int32_t* active_ids, int32_t n_active, void* stream) {
  NvtxRange nvtx_range("rkv:begin_step");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!active_ids || n_active < 1 || n_active > h->cfg.n_streams)
    return fail(h, RKV_ERR_INVALID_ARG, "active_ids must list 1 .. n_streams streams");
  if (h->step_open) {
    const bool exact = rkv::exact_scheme(h->cfg.scheme);
    for (int l = 0; l < h->cfg.n_layers; ++l)
      if (!h->appended[l] || (exact && !h->rebased[l]))
        return fail(h, RKV_ERR_STATE, "previous step left a layer without rkv_append_rope (or rkv_rebase)");
  }
  rkv::ActiveIds ids;
  ids.n = n_active;
  std::vector<uint8_t> seen(h->cfg.n_streams, 0);
  for (int i = 0; i < n_active; ++i) {
    const int32_t s = active_ids[i];
    if (s < 0 || s >= h->cfg.n_streams) return fail(h, RKV_ERR_INVALID_ARG, "stream id out of range");
    if (seen[s]) return fail(h, RKV_ERR_INVALID_ARG, "stream id listed twice");
    seen[s] = 1;
    ids.id[i] = s;
  }
  cudaError_t e = rkv::launch_begin_step(h->view, ids, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "begin_step launch");
  h->step_open = true;
  h->launched_since_begin = false;
  h->n_active = n_active;
  std::fill(h->appended.begin(), h->appended.end(), 0);
  std::fill(h->rebased.begin(), h->rebased.end(), 0);
  return RKV_OK;
}

int rkv_append_rope(rkv_handle* h, int32_t layer, const rkv_bf16* k, const rkv_bf16* v, void* stream) {
  NvtxRange nvtx_range("rkv:append_rope");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (!check_layer(h, layer)) return fail(h, RKV_ERR_INVALID_ARG, "layer out of range");
  if (!k || !v || !aligned16(k) || !aligned16(v))
    return fail(h, RKV_ERR_INVALID_ARG, "k and v must be non-NULL and 16-byte aligned");
  if (h->appended[layer]) return fail(h, RKV_ERR_STATE, "rkv_append_rope called twice for this layer in this step");
  cudaError_t e = rkv::launch_append_rope(h->view, h->n_active, layer, 1, k, v, 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "append_rope launch");
  h->appended[layer] = 1;
  h->launched_since_begin = true;
  return RKV_OK;
}

int rkv_rebase(rkv_handle* h, int32_t layer, void* stream) {
  NvtxRange nvtx_range("rkv:rebase");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!rkv::exact_scheme(h->cfg.scheme)) return fail(h, RKV_ERR_STATE, "rkv_rebase needs an exact re-base scheme");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (!check_layer(h, layer)) return fail(h, RKV_ERR_INVALID_ARG, "layer out of range");
  if (h->rebased[layer]) return fail(h, RKV_ERR_STATE, "rkv_rebase called twice for this layer in this step");
  cudaError_t e = rkv::launch_rebase(h->view, h->n_active, layer, 1, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "rebase launch");
  h->rebased[layer] = 1;
  if (h->cfg.scheme == RKV_SCHEME_EXACT_REBASE) h->launched_since_begin = true;
  return RKV_OK;
}

int rkv_decode_attn(rkv_handle* h, int32_t layer, const rkv_bf16* q, rkv_bf16* out, float* lse, void* stream) {
  NvtxRange nvtx_range("rkv:decode_attn");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (!check_layer(h, layer)) return fail(h, RKV_ERR_INVALID_ARG, "layer out of range");
  if (!q || !out || !aligned16(q) || !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return fail(h, RKV_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (!h->appended[layer]) return fail(h, RKV_ERR_STATE, "rkv_decode_attn before rkv_append_rope for this layer");
  if (rkv::exact_scheme(h->cfg.scheme) && !h->rebased[layer])
    return fail(h, RKV_ERR_STATE, "rkv_decode_attn before rkv_rebase for this layer");
  rkv::AttnExtras x;
  x.early = early_bits(h, false);
  cudaError_t e = rkv::launch_decode_attn(h->view, h->n_active, layer, 1, q, out, lse, 0, 0, x,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "decode_attn launch");
  h->launched_since_begin = true;
  return RKV_OK;
}

int rkv_append_decode_attn(rkv_handle* h, int32_t layer, const rkv_bf16* q, const rkv_bf16* k, const rkv_bf16* v,
                           rkv_bf16* out, float* lse, void* stream) {
  NvtxRange nvtx_range("rkv:append_decode_attn");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (!check_layer(h, layer)) return fail(h, RKV_ERR_INVALID_ARG, "layer out of range");
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return fail(h, RKV_ERR_INVALID_ARG, "q, k, v and out must be non-NULL and 16-byte aligned");
  if (h->appended[layer]) return fail(h, RKV_ERR_STATE, "this layer's tokens were already appended in this step");
  if (rkv::exact_scheme(h->cfg.scheme) && !h->rebased[layer])
    return fail(h, RKV_ERR_STATE, "rkv_append_decode_attn before rkv_rebase for this layer");
  rkv::AttnExtras x;
  x.early = early_bits(h, false);
  x.k_new = k;
  x.v_new = v;
  cudaError_t e = rkv::launch_decode_attn(h->view, h->n_active, layer, 1, q, out, lse, 0, 0, x,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "append_decode_attn launch");
  h->appended[layer] = 1;
  h->launched_since_begin = true;
  return RKV_OK;
}

int rkv_decode_attn_layers(rkv_handle* h, int32_t layer0, int32_t n_layers, const rkv_bf16* q, rkv_bf16* out,
                           float* lse, void* stream) {
  NvtxRange nvtx_range("rkv:decode_attn_layers");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (n_layers < 1 || layer0 < 0 || layer0 + n_layers > h->cfg.n_layers)
    return fail(h, RKV_ERR_INVALID_ARG, "layer range outside [0, n_layers)");
  if (!q || !out || !aligned16(q) || !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return fail(h, RKV_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  const bool exact = rkv::exact_scheme(h->cfg.scheme);
  for (int l = layer0; l < layer0 + n_layers; ++l)
    if (!h->appended[l] || (exact && !h->rebased[l]))
      return fail(h, RKV_ERR_STATE, "rkv_decode_attn_layers before rkv_append_rope (or rkv_rebase) of a layer");
  const rkv_config& c = h->cfg;
  const int64_t rows = static_cast<int64_t>(h->n_active) * c.q_per_step;
  rkv::AttnExtras x;
  x.early = early_bits(h, false);
  cudaError_t e = rkv::launch_decode_attn(h->view, h->n_active, layer0, n_layers, q, out, lse,
                                          rows * c.n_q_heads * c.head_dim, rows * c.n_q_heads, x,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "decode_attn launch");
  h->launched_since_begin = true;
  return RKV_OK;
}

int rkv_step(rkv_handle* h, const int32_t* active_ids, int32_t n_active, const rkv_bf16* q, const rkv_bf16* k,
             const rkv_bf16* v, rkv_bf16* out, float* lse, void* stream) {
  NvtxRange nvtx_range("rkv:step");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return fail(h, RKV_ERR_INVALID_ARG, "q, k, v and out must be non-NULL and 16-byte aligned");
  int rc = rkv_begin_step(h, active_ids, n_active, stream);
  if (rc != RKV_OK) return rc;
  const rkv_config& c = h->cfg;
  const int64_t rows = static_cast<int64_t>(n_active) * c.q_per_step;
  const int64_t q_stride = rows * c.n_q_heads * c.head_dim, kv_stride = rows * c.n_kv_heads * c.head_dim;
  const int64_t lse_stride = rows * c.n_q_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (c.scheme == RKV_SCHEME_EXACT_REBASE) {
    e = rkv::launch_rebase(h->view, n_active, 0, c.n_layers, st);
    if (e != cudaSuccess) return cuda_fail(h, e, "rebase launch");
    h->launched_since_begin = true;
  }
  std::fill(h->rebased.begin(), h->rebased.end(), 1);
  e = rkv::launch_append_rope(h->view, n_active, 0, c.n_layers, k, v, kv_stride, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "append_rope launch");
  h->launched_since_begin = true;
  // q was written before this call, two or more launches back, so the attention kernel may read
  // it before its dependency wait
  rkv::AttnExtras x;
  x.early = early_bits(h, true);
  e = rkv::launch_decode_attn(h->view, n_active, 0, c.n_layers, q, out, lse, q_stride, lse_stride, x, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "decode_attn launch");
  std::fill(h->appended.begin(), h->appended.end(), 1);
  h->launched_since_begin = true;
  return RKV_OK;
}

int rkv_reset_stream(rkv_handle* h, int32_t stream_id, int64_t start_offset, void* stream) {
  NvtxRange nvtx_range("rkv:reset_stream");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (stream_id < 0 || stream_id >= h->cfg.n_streams) return fail(h, RKV_ERR_INVALID_ARG, "stream id out of range");
  if (start_offset < 0 || start_offset >= (int64_t(1) << 52))
    return fail(h, RKV_ERR_CONFIG, "start_offset must be in [0, 2^52)");
  cudaError_t e = rkv::launch_reset_stream(h->view, stream_id, start_offset, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "reset_stream launch");
}

int rkv_reset_streams(rkv_handle* h, const int32_t* ids_dev, const int64_t* p0_dev, int32_t n, void* stream) {
  NvtxRange nvtx_range("rkv:reset_streams");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (n < 0 || n > RKV_MAX_STREAMS || (n > 0 && (!ids_dev || !p0_dev)))
    return fail(h, RKV_ERR_INVALID_ARG, "n must be in [0, RKV_MAX_STREAMS] with non-NULL lists");
  cudaError_t e = rkv::launch_reset_streams(h->view, ids_dev, p0_dev, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "reset_streams launch");
}

namespace {

constexpr int64_t kSnapMagic = 0x31504e5356524bLL;  // "KRVSNP1" little-endian tag
constexpr int kSnapHeader = 16;                    // int64 words of the header
constexpr int kSnapState = rkv::kStateFields;

void snap_header(const rkv_handle* h, int32_t s, int64_t* hdr) {
  const rkv_config& c = h->cfg;
  const int64_t fields[kSnapHeader] = {kSnapMagic, 1, c.n_layers, c.n_kv_heads, c.head_dim, c.page_size,
                                       c.scheme, c.q_per_step, c.rebase_interval,
                                       static_cast<int64_t>(h->n_pages_of[s]), h->regions, c.window_slack,
                                       c.kv_format, 0, 0, 0};
  std::memcpy(hdr, fields, sizeof fields);
}

// Bytes per row (one token, one kv head) of plane r: d 16-bit elements; with the fp8 store d
// bytes of keys or values, and the row's two float scales.
size_t plane_row_bytes(const rkv_handle* h, int r) {
  const rkv_config& c = h->cfg;
  if (c.kv_format != RKV_KV_E4M3) return static_cast<size_t>(c.head_dim) * sizeof(uint16_t);
  return r < 2 ? static_cast<size_t>(c.head_dim) : 2 * sizeof(float);
}

// bytes of one (plane, layer) run of a stream's pages
size_t snap_run_bytes(const rkv_handle* h, int32_t s, int r) {
  const rkv_config& c = h->cfg;
  return static_cast<size_t>(h->n_pages_of[s]) * c.n_kv_heads * c.page_size * plane_row_bytes(h, r);
}

size_t snap_bytes(const rkv_handle* h, int32_t s) {
  size_t b = (kSnapHeader + kSnapState) * sizeof(int64_t);
  for (int r = 0; r < h->regions; ++r) b += static_cast<size_t>(h->cfg.n_layers) * snap_run_bytes(h, s, r);
  return b;
}

// pointer to (plane r, layer l) of stream s's pages
char* snap_run(const rkv_handle* h, int32_t s, int r, int l) {
  const rkv_config& c = h->cfg;
  const size_t rows_per_plane = h->region_elems / c.head_dim, rows_per_layer = h->view.layer_stride / c.head_dim;
  size_t base = 0;
  for (int p = 0; p < r; ++p) base += rows_per_plane * plane_row_bytes(h, p);
  return h->pool + base +
         (static_cast<size_t>(l) * rows_per_layer + static_cast<size_t>(h->first_page[s]) * c.n_kv_heads * c.page_size) *
             plane_row_bytes(h, r);
}

}  // namespace

int rkv_stream_snapshot_bytes(const rkv_handle* h, int32_t stream_id, size_t* bytes) {
  if (!h || !bytes) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle or bytes is NULL");
  if (stream_id < 0 || stream_id >= h->cfg.n_streams) return fail(nullptr, RKV_ERR_INVALID_ARG, "stream id out of range");
  *bytes = snap_bytes(h, stream_id);
  return RKV_OK;
}

int rkv_save_stream(rkv_handle* h, int32_t stream_id, void* dst, size_t bytes, void* stream) {
  NvtxRange nvtx_range("rkv:save_stream");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (stream_id < 0 || stream_id >= h->cfg.n_streams || !dst) return fail(h, RKV_ERR_INVALID_ARG, "bad stream id or dst");
  if (bytes < snap_bytes(h, stream_id)) return fail(h, RKV_ERR_CAPACITY, "dst smaller than rkv_stream_snapshot_bytes");
  if (step_in_progress(h)) return fail(h, RKV_ERR_STATE, "a step is in progress (a layer lacks rkv_append_rope or rkv_rebase)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int64_t hdr[kSnapHeader];
  snap_header(h, stream_id, hdr);
  char* d = static_cast<char*>(dst);
  cudaError_t e = cudaMemcpyAsync(d, hdr, sizeof hdr, cudaMemcpyDefault, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(d + sizeof hdr, h->view.state + static_cast<int64_t>(stream_id) * rkv::kStateFields,
                        kSnapState * sizeof(int64_t), cudaMemcpyDefault, st);
  size_t off = (kSnapHeader + kSnapState) * sizeof(int64_t);
  for (int r = 0; r < h->regions && e == cudaSuccess; ++r) {
    const size_t run = snap_run_bytes(h, stream_id, r);
    for (int l = 0; l < h->cfg.n_layers && e == cudaSuccess; ++l, off += run)
      e = cudaMemcpyAsync(d + off, snap_run(h, stream_id, r, l), run, cudaMemcpyDefault, st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "saving a stream");
}

int rkv_load_stream(rkv_handle* h, int32_t stream_id, const void* src, size_t bytes, void* stream) {
  NvtxRange nvtx_range("rkv:load_stream");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (stream_id < 0 || stream_id >= h->cfg.n_streams || !src) return fail(h, RKV_ERR_INVALID_ARG, "bad stream id or src");
  if (bytes < snap_bytes(h, stream_id)) return fail(h, RKV_ERR_CAPACITY, "src smaller than rkv_stream_snapshot_bytes");
  if (step_in_progress(h)) return fail(h, RKV_ERR_STATE, "a step is in progress (a layer lacks rkv_append_rope or rkv_rebase)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* sp = static_cast<const char*>(src);
  int64_t hdr[kSnapHeader], want[kSnapHeader], state[kSnapState];
  cudaError_t e = cudaMemcpyAsync(hdr, sp, sizeof hdr, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(state, sp + sizeof hdr, sizeof state, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "reading a snapshot header");
  snap_header(h, stream_id, want);
  if (std::memcmp(hdr, want, sizeof hdr) != 0)
    return fail(h, RKV_ERR_CONFIG, "snapshot taken under another configuration, window or scheme");
  if (rkv_check_stream_state(&h->cfg, state) != RKV_OK)
    return fail(h, RKV_ERR_CONFIG, std::string("snapshot state is inconsistent: ") + g_last_error);
  // the window is part of the stream's layout: it must be the slot's own
  int64_t w_dev = 0;
  e = cudaMemcpyAsync(&w_dev, h->view.state + static_cast<int64_t>(stream_id) * rkv::kStateFields + rkv::F_W,
                      sizeof w_dev, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "reading the stream's window");
  if (w_dev != state[rkv::F_W]) return fail(h, RKV_ERR_CONFIG, "snapshot window differs from the stream's window");
  e = cudaMemcpyAsync(h->view.state + static_cast<int64_t>(stream_id) * rkv::kStateFields, sp + sizeof hdr,
                      kSnapState * sizeof(int64_t), cudaMemcpyDefault, st);
  size_t off = (kSnapHeader + kSnapState) * sizeof(int64_t);
  for (int r = 0; r < h->regions && e == cudaSuccess; ++r) {
    const size_t run = snap_run_bytes(h, stream_id, r);
    for (int l = 0; l < h->cfg.n_layers && e == cudaSuccess; ++l, off += run)
      e = cudaMemcpyAsync(snap_run(h, stream_id, r, l), sp + off, run, cudaMemcpyDefault, st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "loading a stream");
}

int rkv_check_stream_state(const rkv_config* cfg, const int64_t* st) {
  std::string why;
  if (!cfg || !st) return fail(nullptr, RKV_ERR_INVALID_ARG, "config or state is NULL");
  if (!validate_config(cfg, &why)) return fail(nullptr, RKV_ERR_CONFIG, why);
  const int64_t n = st[rkv::F_N], len = st[rkv::F_LEN], ev = st[rkv::F_EVICTED], off = st[rkv::F_KV_POS_OFFSET];
  const int64_t rb = st[rkv::F_ROPE_BASE], head = st[rkv::F_HEAD_SLOT], w = st[rkv::F_W], p0 = st[rkv::F_P0];
  const int64_t kMaxPos = int64_t(1) << 52;
  auto bad = [&](const char* m) { return fail(nullptr, RKV_ERR_CONFIG, m); };
  if (w < cfg->q_per_step || w > RKV_MAX_WINDOW) return bad("window outside [q_per_step, RKV_MAX_WINDOW]");
  if (p0 < 0 || p0 >= kMaxPos) return bad("P0 outside [0, 2^52)");
  if (n < 0 || n % cfg->q_per_step != 0 || n >= kMaxPos - p0) return bad("token count n negative, not a multiple of q_per_step, or past 2^52");
  // len as the steps leave it: n until the first step past the ring capacity C = W + slack
  // (which takes n to n1, the first multiple of Q above C, and len to W), then W + k Q with k
  // counting the steps since the last batch, k <= K = floor((C - W) / Q)
  const int64_t q = cfg->q_per_step, ring = w + cfg->window_slack;
  const int64_t n1 = (ring / q + 1) * q;
  const int64_t want_len = n < n1 ? n : w + ((n - n1) / q % ((ring - w) / q + 1)) * q;
  if (len != want_len) return bad("len differs from the eviction rule (min(n, W) without window slack)");
  if (ev != n - len) return bad("evicted differs from n - len");
  if (off != p0 + ev) return bad("kv_pos_offset differs from P0 + evicted");
  if (head != ev % ring) return bad("head_slot differs from evicted mod (W + window_slack)");
  if (rkv::exact_scheme(cfg->scheme)) {
    if (rb < 0 || rb > ev || ev - rb >= cfg->rebase_interval)
      return bad("rope_base outside (evicted - rebase_interval, evicted]");
  } else if (rb != 0) {
    return bad("rope_base must be 0 in the offset-only scheme");
  }
  return RKV_OK;
}

int rkv_get_stream_state(rkv_handle* h, int32_t stream_id, int64_t* out, void* stream) {
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!out || stream_id < 0 || stream_id >= h->cfg.n_streams) return fail(h, RKV_ERR_INVALID_ARG, "bad stream id or out");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, h->view.state + static_cast<int64_t>(stream_id) * rkv::kStateFields,
                                  rkv::kStateFields * sizeof(int64_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "reading stream state");
}

int rkv_sync_status(rkv_handle* h, void* stream) {
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t status[4];
  cudaError_t e = cudaMemcpyAsync(status, h->view.status, sizeof status, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "reading the status word");
  if (status[0] == rkv::DEV_OK) return RKV_OK;
  e = cudaMemsetAsync(h->view.status, 0, sizeof status, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(h, e, "clearing the status word");
  char buf[160];
  const char* what = status[0] == rkv::DEV_TIMEOUT ? "a timed-out wait"
                     : status[0] == rkv::DEV_RANGE ? "a rotated key outside the fp16 range"
                                                   : "an index out of bounds";
  snprintf(buf, sizeof buf, "device reported %s (site %d, value %d)", what, status[1], status[2]);
  const int code = status[0] == rkv::DEV_TIMEOUT ? RKV_ERR_TIMEOUT
                   : status[0] == rkv::DEV_RANGE ? RKV_ERR_DEVICE_RANGE
                                                 : RKV_ERR_DEVICE_BOUNDS;
  return fail(h, code, buf);
}

const char* rkv_last_error(const rkv_handle* h) { return h ? h->last_error.c_str() : g_last_error.c_str(); }

int rkv_destroy(rkv_handle* h) {
  delete h;
  return RKV_OK;
}

int rkv_rope_cossin(const int64_t* pos_dev, int32_t n, int32_t head_dim, double theta, float* cs_dev, void* stream) {
  if (n < 0 || (n > 0 && (!pos_dev || !cs_dev))) return fail(nullptr, RKV_ERR_INVALID_ARG, "bad pointers or n");
  if (head_dim < 2 || head_dim > 128 || head_dim % 2) return fail(nullptr, RKV_ERR_CONFIG, "head_dim must be even, <= 128");
  if (!(theta > 1.0) || !std::isfinite(theta)) return fail(nullptr, RKV_ERR_CONFIG, "theta must be finite and > 1");
  rkv::Omegas w;
  for (int i = 0; i < head_dim / 2; ++i) w.w[i] = std::pow(theta, -2.0 * i / head_dim);
  cudaError_t e = rkv::launch_rope_cossin(pos_dev, n, head_dim, w, cs_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RKV_OK : cuda_fail(nullptr, e, "rope_cossin launch");
}

int rkv_gen_tokens(uint64_t seed, uint32_t tag, int32_t stream_id, int32_t layer, int64_t token0, int32_t n_tokens,
                   int32_t width, float scale, rkv_bf16* out_dev, void* stream) {
  if (n_tokens < 0 || n_tokens > 65535 || width < 0 || (n_tokens && width && !out_dev))
    return fail(nullptr, RKV_ERR_INVALID_ARG, "bad sizes or out pointer");
  cudaError_t e = rkv::launch_gen_tokens(seed, tag, stream_id, layer, token0, n_tokens, width, scale, out_dev,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RKV_OK : cuda_fail(nullptr, e, "gen_tokens launch");
}

int rkv_gen_step_inputs(rkv_handle* h, uint64_t seed, int32_t layer, float scale, rkv_bf16* q, rkv_bf16* k,
                        rkv_bf16* v, void* stream) {
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (!q || !k || !v) return fail(h, RKV_ERR_INVALID_ARG, "q, k, v must be non-NULL");
  cudaError_t e = rkv::launch_gen_step_inputs(h->view, h->n_active, seed, layer, scale, q, k, v,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "gen_step_inputs launch");
}

int rkv_set_wait_test(rkv_handle* h, int32_t withhold_stage, uint64_t wait_ns) {
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (withhold_stage < -1) return fail(h, RKV_ERR_INVALID_ARG, "withhold_stage must be -1 or a stage number");
  if (wait_ns != 0 && (wait_ns < 1000 || wait_ns > rkv::kDefaultWaitNs))
    return fail(h, RKV_ERR_INVALID_ARG, "wait_ns must be 0 (default) or in [1 us, 1 s]");
  h->view.wait_ns = wait_ns ? wait_ns : rkv::kDefaultWaitNs;
  h->view.withhold_stage = withhold_stage;
  return RKV_OK;
}

int rkv_gen_next_inputs(rkv_handle* h, uint64_t seed, const int32_t* active_ids, int32_t n_active, float scale,
                        rkv_bf16* q, rkv_bf16* k, rkv_bf16* v, void* stream) {
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!q || !k || !v) return fail(h, RKV_ERR_INVALID_ARG, "q, k, v must be non-NULL");
  if (!active_ids || n_active < 1 || n_active > h->cfg.n_streams)
    return fail(h, RKV_ERR_INVALID_ARG, "active_ids must list 1 .. n_streams streams");
  rkv::ActiveIds ids;
  ids.n = n_active;
  for (int i = 0; i < n_active; ++i) {
    if (active_ids[i] < 0 || active_ids[i] >= h->cfg.n_streams) return fail(h, RKV_ERR_INVALID_ARG, "stream id out of range");
    ids.id[i] = active_ids[i];
  }
  cudaError_t e = rkv::launch_gen_next_inputs(h->view, ids, seed, scale, q, k, v, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? RKV_OK : cuda_fail(h, e, "gen_next_inputs launch");
}

int rkv_decode_attn_static(rkv_handle* h, int32_t layer, const rkv_bf16* q, rkv_bf16* out, float* lse,
                           void* stream) {
  NvtxRange nvtx_range("rkv:decode_attn_static");
  if (!h) return fail(nullptr, RKV_ERR_INVALID_ARG, "handle is NULL");
  if (!h->step_open) return fail(h, RKV_ERR_STATE, "no open step (call rkv_begin_step)");
  if (!check_layer(h, layer)) return fail(h, RKV_ERR_INVALID_ARG, "layer out of range");
  if (!q || !out || !aligned16(q) || !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return fail(h, RKV_ERR_INVALID_ARG, "q and out must be non-NULL and 16-byte aligned");
  if (!h->appended[layer]) return fail(h, RKV_ERR_STATE, "rkv_decode_attn_static before rkv_append_rope for this layer");
  if (rkv::exact_scheme(h->cfg.scheme) && !h->rebased[layer])
    return fail(h, RKV_ERR_STATE, "rkv_decode_attn_static before rkv_rebase for this layer");
  const size_t need = rkv::static_scratch_need(h->view, h->n_active);
  if (need > rkv::static_scratch_floats()) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "rkv_decode_attn_static needs %zu bytes of scratch for %d active streams; the fixed array holds %zu",
             need * sizeof(float), h->n_active, rkv::static_scratch_floats() * sizeof(float));
    return fail(h, RKV_ERR_CAPACITY, buf);
  }
  cudaError_t e =
      rkv::launch_decode_attn_static(h->view, h->n_active, layer, q, out, lse, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "decode_attn_static launch");
  return RKV_OK;
}

}  // extern "C"

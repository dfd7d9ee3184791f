// Internal declarations shared by the librkv.so translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rkv.h"
#include "twopi_split.h"

namespace rkv {

constexpr int kStateFields = RKV_STATE_FIELDS;
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // a bounded device wait gives up after 1 s
// state field indices (order reported by rkv_get_stream_state)
enum { F_N = 0, F_LEN, F_EVICTED, F_KV_POS_OFFSET, F_ROPE_BASE, F_HEAD_SLOT, F_W, F_P0 };

// status word codes written by kernels (first error wins)
enum { DEV_OK = 0, DEV_BOUNDS = 1, DEV_TIMEOUT = 2, DEV_RANGE = 3 };

// Per active stream of the open step, written by the begin-step kernel.
struct StepDesc {
  int64_t n_old;      // tokens before this step
  int64_t evicted;    // tokens out of the window after this step
  int64_t rope_base;  // exact scheme: origin of stored key positions after this step
  int64_t delta;      // exact scheme: re-base amount this step (0: none)
  int32_t stream;     // stream id
  int32_t len;        // window length after this step
  int32_t ring;       // ring capacity C = W + window_slack: token j lives in ring slot j mod C
  int32_t pad;
};

// Device addresses and shape, passed by value to every kernel.
struct DevView {
  int64_t* state;        // [S][8]
  int32_t* page_table;   // [S][max_pages] -> physical page
  StepDesc* desc;        // [S] by active index
  float* cs_new;         // [S][Q][d/2][2] cos/sin of the new keys' stored positions
  float* cs_q;           // [S][Q][d/2][2] cos/sin of the queries' positions (= cs_new except on read)
  float* cs_lap;         // [S][d/2][2] cos/sin of -W * omega (rotate-on-read scheme only)
  float* rope_table;     // [t_rows][d/2][2] cos/sin of r * omega, r < t_rows (materialised exact re-base)
  double* omega;         // [d/2]
  float* part_ml;        // [S][Q*Hq][splits][2] (running max in log2 units, sum)
  float* part_o;         // [S][Q*Hq][splits][d] normalised partial outputs
  int32_t* status;       // [4]: code, detail, detail2, unused
  uint16_t* k_rot;       // pool: [L][n_pages][Hkv][ps][d] rotated keys, fp16 bits
  uint16_t* v;           // pool: values (bf16 bits), same layout
  uint16_t* k_raw;       // pool: pre-RoPE keys (bf16 bits; materialised exact re-base only), same layout
  // fp8 store (kv_format e4m3): k_rot and v point at planes of d bytes per row instead, and
  // kv_scale at the rows' (key, value) scales 2^e, [L][n_pages][Hkv][ps]; NULL otherwise
  float2* kv_scale;
  int64_t layer_stride;  // elements of one layer in one pool region
  int32_t n_streams, n_layers, n_q_heads, n_kv_heads, head_dim, q_per_step;
  int32_t page_size, n_pages, max_pages, t_rows;
  int32_t scheme, rebase_interval, window_slack;
  int32_t num_sms;       // host-side launch planning only
  float scale_log2;      // softmax scale * log2(e)
  // failure-detection test hook (rkv_set_wait_test): bounded waits give up after wait_ns; the
  // attention producer skips the copy of its stage number withhold_stage (-1: none)
  unsigned long long wait_ns;
  int32_t withhold_stage;
};

// Both exact schemes keep window-relative key positions and a rope_base.
__host__ __device__ __forceinline__ bool exact_scheme(int scheme) {
  return scheme == RKV_SCHEME_EXACT_REBASE || scheme == RKV_SCHEME_EXACT_ON_READ;
}

// Pool rows are d 16-bit elements = d/8 chunks of 16 bytes.  Chunk c of the
// row at offset `off` inside its page lives at chunk position c ^ (off & 7):
// eight consecutive rows put any one chunk in eight different shared-memory
// bank groups once a page is copied verbatim into shared memory, so 8x8
// matrix loads (ldmatrix) of the page are conflict-free.
__host__ __device__ __forceinline__ int swizzle_chunk(int chunk, int off) { return chunk ^ (off & 7); }

struct Omegas {
  double w[64];  // omega_i = theta^(-2i/d), i < d/2, rounded to fp64 on the host
};

struct ActiveIds {
  int32_t n;
  int32_t id[RKV_MAX_STREAMS];
};

// Programmatic dependent launch: the hot-path kernels are launched so that the
// next kernel in the stream may be scheduled while this one runs.  Each kernel
// waits for its predecessor to complete (memory visible) and only then lets
// its own dependents launch, so when any of them starts, every kernel two
// launches back has completed: a kernel may read, before its own wait, data
// that only those earlier kernels write (the step descriptors, the page table,
// the caller's queries inside rkv_step, which were written before the call),
// never data its immediate predecessor may write (a caller's kernel that
// writes the queries just before rkv_decode_attn, for instance).  A
// dependent grid launches only after every CTA of its predecessor has
// started, so waiting CTAs never hold resources the predecessor still needs.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void record_error(int32_t* status, int code, int detail, int detail2) {
  if (atomicCAS(status, DEV_OK, code) == DEV_OK) {
    status[1] = detail;
    status[2] = detail2;
  }
}

// cos/sin of p * omega in fp32 from an fp64 computation whose only error is
// the final rounding steps.  p * omega = hi + lo exactly (FMA; |p| < 2^53).
// k = nearest integer to hi / (2 pi).  With 2 pi = C1 + C2 + C3,
// hi - k*C1 is exact under FMA (the result is a multiple of ulp(C1) below 8
// in magnitude), then k*C2, k*C3 and lo are folded in with one rounding each.
__device__ __forceinline__ void rope_cos_sin(int64_t p, double omega, float* c, float* s) {
  const double pd = static_cast<double>(p);
  const double hi = pd * omega;
  const double lo = fma(pd, omega, -hi);
  const double k = rint(hi * RKV_INV_TWO_PI);
  double r = fma(-k, RKV_TWO_PI_C1, hi);
  r = fma(-k, RKV_TWO_PI_C2, r);
  r = fma(-k, RKV_TWO_PI_C3, r);
  r += lo;
  double sd, cd;
  sincos(r, &sd, &cd);
  *c = static_cast<float>(cd);
  *s = static_cast<float>(sd);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// round to nearest, ties to even (finite inputs)
__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// fp32 -> fp16 bits, round to nearest even
__device__ __forceinline__ uint16_t f32_to_f16(float x) { return __half_as_ushort(__float2half_rn(x)); }

__device__ __forceinline__ float f16_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// largest finite fp16 value after rounding: |x| >= 65520 rounds to infinity
__device__ __forceinline__ bool fits_f16(float x) { return fabsf(x) < 65520.0f; }

// ---- fp8 store (kv_format e4m3): rows of d elements, each with a power-of-two scale 2^e, e the
// smallest integer for which max|x| / 2^e <= 448 (the largest finite e4m3 magnitude, 1.75 * 2^8):
// with max|x| = f * 2^E, f in [0.5, 1), that is E - 9 when f <= 0.875 and E - 8 otherwise.  A row
// of zeros takes e = 0; e stays >= -126 so that 2^e is a normal float.
__device__ __forceinline__ int e4m3_row_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int big_e;
  const float f = frexpf(amax, &big_e);
  const int e = f <= 0.875f ? big_e - 9 : big_e - 8;
  return e < -126 ? -126 : e;
}
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

// two fp32 (already divided by the row's 2^e, so within +-448) to e4m3, nearest even: x0 in the
// low byte, x1 in the high byte
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}
// two e4m3 (low byte first) to fp16x2 (low half first), exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t b) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(b));
  return r;
}
// two e4m3 to bf16x2, exact (every e4m3 value is a bf16 value)
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t b) {
  const uint32_t h = e4m3x2_to_f16x2(b);
  const float lo = __half2float(__ushort_as_half(static_cast<uint16_t>(h & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half(static_cast<uint16_t>(h >> 16)));
  return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}
// eight fp32 divided by 2^e to eight e4m3 bytes (element 0 in the lowest byte)
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], float inv_scale) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = f32x2_to_e4m3x2(x[2 * j] * inv_scale, x[2 * j + 1] * inv_scale);
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// element offset of (layer, physical page, kv head, offset in page) in a pool region
__device__ __forceinline__ int64_t pool_offset(const DevView& v, int layer, int page, int kvh, int off) {
  return static_cast<int64_t>(layer) * v.layer_stride +
         ((static_cast<int64_t>(page) * v.n_kv_heads + kvh) * v.page_size + off) * v.head_dim;
}

// ---- launchers (host functions, one translation unit each) ----
cudaError_t launch_init_tables(const DevView& v, cudaStream_t st);
cudaError_t launch_begin_step(const DevView& v, const ActiveIds& ids, cudaStream_t st);
cudaError_t launch_reset_stream(const DevView& v, int s, int64_t p0, cudaStream_t st);
cudaError_t launch_reset_streams(const DevView& v, const int32_t* ids, const int64_t* p0, int n, cudaStream_t st);
// Layers [layer0, layer0 + n_layers) in one launch; per-layer tensors of the
// step's inputs/outputs are `*_layer_stride` elements apart.
cudaError_t launch_append_rope(const DevView& v, int n_active, int layer0, int n_layers, const uint16_t* k,
                               const uint16_t* vv, int64_t kv_layer_stride, cudaStream_t st);
cudaError_t launch_rebase(const DevView& v, int n_active, int layer0, int n_layers, cudaStream_t st);

// How decode attention splits the window of one (layer, stream, kv head).
struct AttnPlan {
  int splits;            // CTAs per (layer, stream, kv head)
  int stages_per_split;  // 64-slot stages each CTA streams
  bool cluster;          // splits merged through distributed shared memory
  int64_t slots;         // CTAs the launch may keep resident (whole windows: grid <= slots)
};
// cluster = true: splits combine in distributed shared memory (no scratch);
// false: every split writes (m, l, o) to part_ml / part_o and a merge kernel
// combines them (single layer only).
AttnPlan plan_decode_attn(const DevView& v, int n_active, int n_layers, bool cluster);
// What a decode-attention launch may read before its dependency wait, and the fused append.
constexpr int kEarlyDesc = 1;  // step descriptors and angles: the begin-step kernel ran two or more launches back
constexpr int kEarlyQ = 2;     // the queries: written before the call that launches (rkv_step)
struct AttnExtras {
  int early = 0;
  const uint16_t* k_new = nullptr;  // fused append: pre-RoPE keys [layer][A][Q][Hkv][d]
  const uint16_t* v_new = nullptr;  // and values, written into the pool by the attention launch
  int64_t kv_layer_stride = 0;
};
cudaError_t launch_decode_attn(const DevView& v, int n_active, int layer0, int n_layers, const uint16_t* q,
                               uint16_t* out, float* lse, int64_t q_layer_stride, int64_t lse_layer_stride,
                               const AttnExtras& x, cudaStream_t st);
// the split-K form with partials in v.part_ml / v.part_o (one layer)
cudaError_t launch_decode_attn_scratch(const DevView& v, int n_active, int layer, const uint16_t* q, uint16_t* out,
                                       float* lse, cudaStream_t st);
// decode attention with its split-K scratch in the library's fixed array (rkv_noalloc.cu)
size_t static_scratch_floats();
size_t static_scratch_need(const DevView& v, int n_active);
cudaError_t launch_decode_attn_static(const DevView& v, int n_active, int layer, const uint16_t* q, uint16_t* out,
                                      float* lse, cudaStream_t st);
cudaError_t launch_rope_cossin(const int64_t* pos, int n, int head_dim, const Omegas& w, float* cs,
                               cudaStream_t st);
cudaError_t launch_gen_tokens(uint64_t seed, uint32_t tag, int32_t stream_id, int32_t layer, int64_t token0,
                              int32_t n_tokens, int32_t width, float scale, uint16_t* out, cudaStream_t st);
cudaError_t launch_gen_next_inputs(const DevView& v, const ActiveIds& ids, uint64_t seed, float scale, uint16_t* q,
                                   uint16_t* k, uint16_t* vv, cudaStream_t st);
cudaError_t launch_gen_step_inputs(const DevView& v, int n_active, uint64_t seed, int32_t layer, float scale,
                                   uint16_t* q, uint16_t* k, uint16_t* vv, cudaStream_t st);

}  // namespace rkv

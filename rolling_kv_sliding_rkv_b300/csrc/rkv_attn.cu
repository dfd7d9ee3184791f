// Windowed GQA decode attention over the ring (Audio8 ASR Infinite
// 无限长转写原理, "Rolling KV Cache 三步拆解", 第 3 步: attention scans only
// the fixed window, so the cost of a step is constant).
//
// One CTA streams the K/V pages of one (layer, stream, kv head), or of a
// contiguous share of them (split-K), through shared memory and keeps an
// online softmax for the kv head's G = Hq/Hkv query heads times the step's Q
// queries (R = G*Q rows, at most 16).
//
// Data movement.  A stage is 64 consecutive ring slots: K and V page blocks
// (64 x d 16-bit values each, contiguous in the pool) land in shared memory
// through bulk asynchronous copies (cp.async.bulk) issued by one producer
// warp and completed on an mbarrier; 96 KB of stages are in flight per CTA
// (three at d = 128, six at d = 64), up to two CTAs per SM.  The pool's chunk
// swizzle (rkv_internal.cuh) makes the verbatim copies conflict-free for
// ldmatrix.
//
// Arithmetic.  Per warp, 16 keys at a time on the tensor cores (mma.sync
// m16n8k16, fp32 accumulate), with keys as the M dimension so the query rows
// fill N = 8 without padding:
//   S^T[16 keys][8 rows] = K[16][d] . Qs^T, Qs = q rotated in fp32, times the
//       softmax scale * log2(e), split into fp16 hi + lo parts (two MMAs), so
//       the query adds no rounding of its own;
//   P^T = exp2(S^T - m) (rows' running max m), rounded to bf16 and turned
//       into the B operand by an 8x8 transpose (movmatrix);
//   O^T[d][8 rows] += V^T[d][16 keys] . P^T  (V read with ldmatrix.trans).
// Stored keys are fp16.  In the exact re-base applied on read, a key is
// stored rotated by its ring slot index (j mod C, C the ring's capacity) and
// never touched again; the query carries the rest of the rotation: for ring
// slots at or above evicted mod C it is rotated to j_q - C * floor(evicted /
// C), for the slots below (tokens of the ring's next lap) C less, so every
// score sees the exact position difference of its tokens.  The second query
// is R(-C) applied to the first, built once per unit in shared memory
// (build_next_lap).
//
// Splits of one (layer, stream, kv head) form a thread-block cluster and
// combine their (m, l, O) through distributed shared memory; the scratch
// form writes per-split partials to global memory for a separate merge.
// Every sum runs in a fixed order, so outputs are reproducible run to run.
//
// With the append fused (rkv_append_decode_attn), a sixth warp writes the
// step's new keys and values into the pool while the others stream the
// window's older stages, which a unit's walk takes first.  With the optional
// fp8 store, stages hold e4m3 codes and their rows' scales; each consumer
// warp expands its 16 rows into a 16-bit stage before the fragment loads.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "rkv_async.cuh"
#include "rkv_internal.cuh"

namespace rkv {
namespace {

constexpr int kCW = 4;                    // consumer warps: 16 slots of every stage each
constexpr int kThreads = (kCW + 1) * 32;  // + one producer warp
// threads of a CTA: with the append fused, a sixth warp writes the step's new tokens
template <bool FUSE>
__host__ __device__ constexpr int threads_of() {
  return FUSE ? kThreads + 32 : kThreads;
}
static_assert(kCW == 4, "the epilogue sums warps 0 + 2 and 1 + 3");
constexpr int kKS = 64;                   // ring slots per stage
// shared-memory ring per CTA: 96 KB of K/V stages whatever the head dim
template <int D>
__host__ __device__ constexpr int stages_for() {
  return 3 * 128 / D;
}

struct AttnArgs {
  DevView v;
  const uint16_t* q;   // [layer][A][Q][Hq][d]
  uint16_t* out;       // [layer][A][Q][Hq][d]
  float* lse;          // [layer][A][Q][Hq] or NULL
  int64_t q_layer_stride, lse_layer_stride;
  int layer0, n_layers, n_active;
  int splits, stages_per_split;
  int mode;            // 0: whole windows; 1: split, cluster merge; 2: split, partials to part_ml / part_o
  // What may be read before the dependency wait (programmatic dependent launch; see
  // rkv_internal.cuh): bit 0 the step descriptors, angles and pages (the begin-step kernel ran two
  // or more launches back), bit 1 the queries (written before the call, rkv_step).  A cleared bit
  // means the data may come from this launch's immediate predecessor and is read after the wait.
  int early;
  // fused append (rkv_append_decode_attn): the step's new keys and values, pre-RoPE,
  // [layer][A][Q][Hkv][d], written rotated into the pool by the CTA's appender warp before the
  // producer copies their stage; NULL when rkv_append_rope did it
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t kv_layer_stride;
};


// 2^x with the hardware approximation (relative error about 2^-22; subnormal
// results flush to zero, which softmax weights below 2^-126 can afford)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory"); }

// consumer_sync that also returns whether any consumer thread passed `pred`
__device__ __forceinline__ bool consumer_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, o;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred o, 1, %2, a;\n\tselp.u32 %0, 1, 0, o;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kCW * 32)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float ld_dsmem_f32(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float x;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(remote) : "memory");
  return x;
}

template <int D, int NT>
__host__ __device__ constexpr int smem_bytes() {
  // stages (K | V), query tiles hi + lo, two fp32 output tiles
  return stages_for<D>() * 2 * kKS * D * 2 + 2 * (8 * NT) * (D + 8) * 2 + 2 * (8 * NT) * (D + 4) * 4;
}

// fp8 store: a stage is 64 rows of fp8 keys, 64 of fp8 values and 64 (key, value) scale pairs;
// ~50 KB of stages (as many tokens in flight as 100 KB of fp16 ones), then one expanded stage
// (K | V in 16 bits, the fp16 stage layout) that the consumer warps fill from each stage; two
// CTAs still fit an SM
template <int D>
__host__ __device__ constexpr int stage8_bytes() {
  return 2 * kKS * D + kKS * 8;
}
template <int D>
__host__ __device__ constexpr int stages8_for() {
  return D == 128 ? 3 : 6;
}
template <int D, int NT, bool KV8>
__host__ __device__ constexpr int smem_bytes_for() {
  return KV8 ? stages8_for<D>() * stage8_bytes<D>() + 2 * kKS * D * 2 + 2 * (8 * NT) * (D + 8) * 2 +
                   2 * (8 * NT) * (D + 4) * 4
             : smem_bytes<D, NT>();
}
static_assert(smem_bytes_for<128, 1, true>() <= 100 * 1024 && smem_bytes_for<64, 1, true>() <= 100 * 1024,
              "two fp8-store CTAs per SM");
static_assert(smem_bytes<128, 2>() <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ float4 ld_dsmem_f32x4(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  float4 x;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
               : "r"(remote)
               : "memory");
  return x;
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8]) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}

// The unit (layer offset, active stream, kv head) of flat index u.
struct Unit {
  int lz, a, kvh;
};
__device__ __forceinline__ Unit unit_of(int u, int n_active, int hkv) {
  Unit r;
  const int per_layer = n_active * hkv;
  r.lz = u / per_layer;
  const int rem = u - r.lz * per_layer;
  r.a = rem / hkv;
  r.kvh = rem - r.a * hkv;
  return r;
}

// Ring slots written so far: all C once anything was evicted, else 0 .. len-1.  With a ring
// capacity above the window (window_slack > 0) some of them hold evicted tokens: masked.
__device__ __forceinline__ int slots_in_use(const StepDesc& d) { return d.evicted > 0 ? d.ring : d.len; }

// Query prefetch of one consumer thread, pair cp of row r (chunks cp and cp + D/16), and, on
// read, element tid of the unit's (cos, sin)(-C omega) row.  The cos/sin of the pair's eight
// frequencies go to registers.  The raw bf16 chunks and the lap element go either to registers
// too, or (STAGED) by cp.async into the thread's own slots of the CTA's raw-query rows and into
// lap_dst, so that those registers are not tied up while the current unit streams: the consumers
// sit at the register limit of two CTAs per SM, and the re-base applied on read, whose lap switch
// needs the most, runs faster staged (the other kernels measured faster without).  The issuing
// thread reads its chunks back after cp_async_wait_all; other threads read the lap row after the
// next barrier.
template <int D>
struct QPrefetch {
  uint4 xa, xb;  // register form only
  float4 cs[4];
  float lap;     // register form only
};

template <int D, bool STAGED>
__device__ __forceinline__ void q_prefetch(const AttnArgs& args, const Unit& un, int tid, QPrefetch<D>& pf,
                                           uint16_t* qraw_s, float* lap_dst) {
  constexpr int CP = D / 16, H = D / 2;
  const DevView& v = args.v;
  const int r = tid / CP, cp = tid % CP;
  const int group = v.n_q_heads / v.n_kv_heads, nq = v.q_per_step;
  if (r < group * nq) {
    const int t = r / group, h = un.kvh * group + r % group;
    const uint16_t* x =
        args.q + un.lz * args.q_layer_stride + ((static_cast<int64_t>(un.a) * nq + t) * v.n_q_heads + h) * D;
    if constexpr (STAGED) {
      cp_async16(qraw_s + r * D + cp * 8, x + cp * 8);
      cp_async16(qraw_s + r * D + H + cp * 8, x + H + cp * 8);
    } else {
      pf.xa = *reinterpret_cast<const uint4*>(x + cp * 8);
      pf.xb = *reinterpret_cast<const uint4*>(x + H + cp * 8);
    }
    const float4* cs = reinterpret_cast<const float4*>(v.cs_q + ((static_cast<int64_t>(un.a) * nq + t) * H + cp * 8) * 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) pf.cs[j] = cs[j];
  } else {
    if constexpr (!STAGED) pf.xa = pf.xb = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) pf.cs[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if constexpr (STAGED) {
    if (lap_dst && tid < D) cp_async4(lap_dst + tid, v.cs_lap + static_cast<int64_t>(un.a) * D + tid);
  } else {
    pf.lap = v.cs_lap && tid < D ? v.cs_lap[static_cast<int64_t>(un.a) * D + tid] : 0.f;
  }
}

// Rotate, scale to log2 units and split into fp16 hi + lo; write the tiles (rows from rows_live
// on are zero).  STAGED: the caller has waited for its own cp.async copies.
template <int D, int NT, bool STAGED>
__device__ __forceinline__ void q_build(const QPrefetch<D>& pf, float scale_log2, int tid, uint16_t* qh_s,
                                        uint16_t* ql_s, const uint16_t* qraw_s, int rows_live) {
  constexpr int CP = D / 16, H = D / 2, QSTR = D + 8;
  const int r = tid / CP, cp = tid % CP;
  if (r >= 8 * NT) return;
  uint4 xa, xb;
  if constexpr (STAGED) {
    const bool live = r < rows_live;
    xa = live ? *reinterpret_cast<const uint4*>(qraw_s + r * D + cp * 8) : make_uint4(0, 0, 0, 0);
    xb = live ? *reinterpret_cast<const uint4*>(qraw_s + r * D + H + cp * 8) : make_uint4(0, 0, 0, 0);
  } else {
    xa = pf.xa;
    xb = pf.xb;
  }
  const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
  const float* cs = reinterpret_cast<const float*>(pf.cs);
  uint32_t ha[4], hb[4], la[4], lb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float ya[2], yb[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float xa = __uint_as_float(e ? (wa[j] & 0xFFFF0000u) : (wa[j] << 16));
      const float xb = __uint_as_float(e ? (wb[j] & 0xFFFF0000u) : (wb[j] << 16));
      const float c = cs[4 * j + 2 * e], s = cs[4 * j + 2 * e + 1];
      ya[e] = (xa * c - xb * s) * scale_log2;
      yb[e] = (xa * s + xb * c) * scale_log2;
    }
    const __half2 hA = __floats2half2_rn(ya[0], ya[1]), hB = __floats2half2_rn(yb[0], yb[1]);
    const float2 fA = __half22float2(hA), fB = __half22float2(hB);
    ha[j] = *reinterpret_cast<const uint32_t*>(&hA);
    hb[j] = *reinterpret_cast<const uint32_t*>(&hB);
    la[j] = pack_f16(ya[0] - fA.x, ya[1] - fA.y);
    lb[j] = pack_f16(yb[0] - fB.x, yb[1] - fB.y);
  }
  *reinterpret_cast<uint4*>(qh_s + r * QSTR + cp * 8) = make_uint4(ha[0], ha[1], ha[2], ha[3]);
  *reinterpret_cast<uint4*>(qh_s + r * QSTR + H + cp * 8) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
  *reinterpret_cast<uint4*>(ql_s + r * QSTR + cp * 8) = make_uint4(la[0], la[1], la[2], la[3]);
  *reinterpret_cast<uint4*>(ql_s + r * QSTR + H + cp * 8) = make_uint4(lb[0], lb[1], lb[2], lb[3]);
}

// ---------------- exact re-base applied on read: the query of the ring's next lap
//
// Built once per unit by the four consumer warps together, from the current lap's tiles: every
// element pair (i, i + d/2) of every query row is rebuilt in fp32 from its hi + lo parts, rotated
// with (cos, sin)(-C omega_i) and split into fp16 hi + lo again (a relative error of a few 2^-24,
// far below the fp16 rounding of a stored key).  Two adjacent frequencies per item.
template <int D, int NT>
__device__ __forceinline__ void build_next_lap(const uint16_t* qh_s, const uint16_t* ql_s, uint16_t* bh_s,
                                               uint16_t* bl_s, const float* lap, int tid) {
  constexpr int QSTR = D + 8, H = D / 2, ITEMS = 8 * NT * (D / 4);
  for (int it = tid; it < ITEMS; it += kCW * 32) {
    const int r = it / (D / 4), i = (it % (D / 4)) * 2;
    const int oa = r * QSTR + i, ob = oa + H;
    const float2 ah = __half22float2(*reinterpret_cast<const __half2*>(qh_s + oa));
    const float2 al = __half22float2(*reinterpret_cast<const __half2*>(ql_s + oa));
    const float2 bh = __half22float2(*reinterpret_cast<const __half2*>(qh_s + ob));
    const float2 bl = __half22float2(*reinterpret_cast<const __half2*>(ql_s + ob));
    const float4 cs = *reinterpret_cast<const float4*>(lap + 2 * i);  // (cos, sin) of i, i + 1
    const float a0 = ah.x + al.x, a1 = ah.y + al.y, b0 = bh.x + bl.x, b1 = bh.y + bl.y;
    const float ra0 = a0 * cs.x - b0 * cs.y, rb0 = a0 * cs.y + b0 * cs.x;
    const float ra1 = a1 * cs.z - b1 * cs.w, rb1 = a1 * cs.w + b1 * cs.z;
    const __half2 ha = __floats2half2_rn(ra0, ra1), hb = __floats2half2_rn(rb0, rb1);
    const float2 fa = __half22float2(ha), fb = __half22float2(hb);
    *reinterpret_cast<__half2*>(bh_s + oa) = ha;
    *reinterpret_cast<__half2*>(bh_s + ob) = hb;
    *reinterpret_cast<uint32_t*>(bl_s + oa) = pack_f16(ra0 - fa.x, ra1 - fa.y);
    *reinterpret_cast<uint32_t*>(bl_s + ob) = pack_f16(rb0 - fb.x, rb1 - fb.y);
  }
}

// Fused append (rkv_append_decode_attn): a sixth warp of the CTA, the appender, writes the step's
// new tokens of every (layer, stream, kv head) the CTA walks into the pool, as rkv_append_rope would
// write them (key rotated by its cos/sin row and rounded to fp16, the pre-RoPE key for the
// materialised re-base, the value as given), while the producer streams the window's older stages.
// The walk of a unit then starts at the stage after the one holding its newest token, so that the
// stages with new rows come last and their bulk copies, which wait for the appender, find its
// rows written.  Position i of a unit's walk is stage (rot + i) mod n_st.
// Ring slot of new token t, from the slot of the step's first (one 64-bit remainder per unit).
__device__ __forceinline__ int first_new_slot(const StepDesc& dsc) { return static_cast<int>(dsc.n_old % dsc.ring); }
__device__ __forceinline__ int new_slot(int first, int t, int ring) {
  const int s = first + t;
  return s >= ring ? s - ring : s;
}

__device__ __forceinline__ int walk_rot(int first, int nq, int ring, int n_st) {
  if (n_st <= 0) return 0;
  const int last = new_slot(first, nq - 1, ring) / kKS;
  return last + 1 >= n_st ? 0 : last + 1;
}

__device__ __forceinline__ bool stage_has_new(int first, int nq, int ring, int st) {
  for (int t = 0; t < nq; ++t)
    if (new_slot(first, t, ring) / kKS == st) return true;
  return false;
}

// New token t of the unit into the pool: lane c < D/16 rotates chunk pair (c, c + D/16) of its
// key, lanes D/16 .. D/16 + D/8 - 1 copy one 16-byte chunk of its value.
template <int D>
__device__ __forceinline__ void append_token(const AttnArgs& args, const StepDesc& dsc, const Unit& un, int t,
                                             int slot, int lane) {
  const DevView& v = args.v;
  const int nq = v.q_per_step, hkv = v.n_kv_heads, ps = v.page_size;
  const int layer = args.layer0 + un.lz;
  constexpr int CP = D / 16, H = D / 2;
  const int rp = slot / ps, off = slot % ps;
  const int page = rp < v.max_pages ? v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + rp] : -1;
  if (page < 0 || page >= v.n_pages) {
    if (lane == 0) record_error(v.status, DEV_BOUNDS, 24, page);
    return;
  }
  const int64_t dst = pool_offset(v, layer, page, un.kvh, off);
  const int64_t row = static_cast<int64_t>(un.a) * nq + t;
  const int64_t src = un.lz * args.kv_layer_stride + (row * hkv + un.kvh) * D;
  if (lane < CP) {
    const int c = lane;
    const uint4 ka = *reinterpret_cast<const uint4*>(args.k_new + src + c * 8);
    const uint4 kb = *reinterpret_cast<const uint4*>(args.k_new + src + H + c * 8);
    const float4* cs = reinterpret_cast<const float4*>(v.cs_new + (row * H + c * 8) * 2);
    const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
    uint32_t ya[4], yb[4];
    bool ok = true;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 rc = cs[j];  // (cos, sin) of elements 2j, 2j + 1 of the chunk
      const float a0 = __uint_as_float(wa[j] << 16), a1 = __uint_as_float(wa[j] & 0xFFFF0000u);
      const float b0 = __uint_as_float(wb[j] << 16), b1 = __uint_as_float(wb[j] & 0xFFFF0000u);
      const float ra0 = a0 * rc.x - b0 * rc.y, rb0 = a0 * rc.y + b0 * rc.x;
      const float ra1 = a1 * rc.z - b1 * rc.w, rb1 = a1 * rc.w + b1 * rc.z;
      ok = ok && fits_f16(ra0) && fits_f16(ra1) && fits_f16(rb0) && fits_f16(rb1);
      ya[j] = pack_f16(ra0, ra1);
      yb[j] = pack_f16(rb0, rb1);
    }
    if (!ok) record_error(v.status, DEV_RANGE, 3, c);
    const int pa = swizzle_chunk(c, off) * 8, pb = swizzle_chunk(c + CP, off) * 8;
    *reinterpret_cast<uint4*>(v.k_rot + dst + pa) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    *reinterpret_cast<uint4*>(v.k_rot + dst + pb) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
    if (v.k_raw) {
      *reinterpret_cast<uint4*>(v.k_raw + dst + pa) = ka;
      *reinterpret_cast<uint4*>(v.k_raw + dst + pb) = kb;
    }
  } else if (lane < CP + D / 8) {
    const int c = lane - CP;
    const uint4 x = *reinterpret_cast<const uint4*>(args.v_new + src + c * 8);
    *reinterpret_cast<uint4*>(v.v + dst + swizzle_chunk(c, off) * 8) = x;
  }
}

// The same token into the fp8 store: key lanes c < D/16 rotate chunk pair (c, c + D/16), value
// lanes VB .. VB + D/8 - 1 hold one chunk of 8 values (VB = D/8, so that each group is an aligned
// run of lanes); butterflies give each group its row's largest magnitude, and the codes of x / 2^e
// go to the row's bytes, the scales beside.  Every lane of the warp calls it.
template <int D>
__device__ __forceinline__ void append_token_e4m3(const AttnArgs& args, const StepDesc& dsc, const Unit& un, int t,
                                                  int slot, int lane) {
  const DevView& v = args.v;
  const int nq = v.q_per_step, hkv = v.n_kv_heads, ps = v.page_size;
  const int layer = args.layer0 + un.lz;
  constexpr int CP = D / 16, H = D / 2, VB = D / 8;
  const int rp = slot / ps, off = slot % ps;
  const int page = rp < v.max_pages ? v.page_table[static_cast<int64_t>(dsc.stream) * v.max_pages + rp] : -1;
  if (page < 0 || page >= v.n_pages) {
    if (lane == 0) record_error(v.status, DEV_BOUNDS, 24, page);
    return;
  }
  const int64_t dst = pool_offset(v, layer, page, un.kvh, off);  // row index * D: a byte offset here
  const int64_t row = static_cast<int64_t>(un.a) * nq + t;
  const int64_t src = un.lz * args.kv_layer_stride + (row * hkv + un.kvh) * D;
  float ra[8], rb[8];
  float km = 0.f, vm = 0.f;
  if (lane < CP) {
    const uint4 ka = *reinterpret_cast<const uint4*>(args.k_new + src + lane * 8);
    const uint4 kb = *reinterpret_cast<const uint4*>(args.k_new + src + H + lane * 8);
    const float4* cs = reinterpret_cast<const float4*>(v.cs_new + (row * H + lane * 8) * 2);
    const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
    bool ok = true;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 rc = cs[j];
      const float a0 = __uint_as_float(wa[j] << 16), a1 = __uint_as_float(wa[j] & 0xFFFF0000u);
      const float b0 = __uint_as_float(wb[j] << 16), b1 = __uint_as_float(wb[j] & 0xFFFF0000u);
      // every product and sum rounded to fp32 on its own, as the append kernel does
      ra[2 * j] = __fsub_rn(__fmul_rn(a0, rc.x), __fmul_rn(b0, rc.y));
      rb[2 * j] = __fadd_rn(__fmul_rn(a0, rc.y), __fmul_rn(b0, rc.x));
      ra[2 * j + 1] = __fsub_rn(__fmul_rn(a1, rc.z), __fmul_rn(b1, rc.w));
      rb[2 * j + 1] = __fadd_rn(__fmul_rn(a1, rc.w), __fmul_rn(b1, rc.z));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ok = ok && fits_f16(ra[j]) && fits_f16(rb[j]);
      km = fmaxf(km, fmaxf(fabsf(ra[j]), fabsf(rb[j])));
    }
    if (!ok) record_error(v.status, DEV_RANGE, 3, lane);
  } else if (lane >= VB && lane < VB + D / 8) {
    const uint4 x = *reinterpret_cast<const uint4*>(args.v_new + src + (lane - VB) * 8);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      ra[2 * j] = __uint_as_float(w[j] << 16);
      ra[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) vm = fmaxf(vm, fabsf(ra[j]));
    // read back as fp16 code * 2^e: a row must stay clear of the fp16 limit after rounding up a code
    if (!(vm < 61440.f)) record_error(v.status, DEV_RANGE, 4, lane);
  }
#pragma unroll
  for (int o = 1; o < D / 8; o <<= 1) {  // key groups of CP lanes and value groups of D/8, aligned
    const float pk = __shfl_xor_sync(0xffffffffu, km, o), pv = __shfl_xor_sync(0xffffffffu, vm, o);
    if (o < CP) km = fmaxf(km, pk);
    vm = fmaxf(vm, pv);
  }
  const int ek = e4m3_row_exponent(__shfl_sync(0xffffffffu, km, 0));
  const int ev = e4m3_row_exponent(__shfl_sync(0xffffffffu, vm, VB));
  uint8_t* k8 = reinterpret_cast<uint8_t*>(v.k_rot);
  uint8_t* v8 = reinterpret_cast<uint8_t*>(v.v);
  if (lane < CP) {
    *reinterpret_cast<uint2*>(k8 + dst + lane * 8) = quantize8(ra, exp2_int(-ek));
    *reinterpret_cast<uint2*>(k8 + dst + H + lane * 8) = quantize8(rb, exp2_int(-ek));
    if (lane == 0) v.kv_scale[dst / D] = make_float2(exp2_int(ek), exp2_int(ev));
  } else if (lane >= VB && lane < VB + D / 8) {
    *reinterpret_cast<uint2*>(v8 + dst + (lane - VB) * 8) = quantize8(ra, exp2_int(-ev));
  }
}

// Up to two CTAs per SM.  Without a cluster the CTA walks units u = blockIdx.x,
// blockIdx.x + gridDim.x, ... (whole windows, no split), its producer warp
// streaming the next unit's pages while the consumers finish the current
// one.  With a cluster (few units, window split over `splits` CTAs) every
// CTA takes exactly one (unit, split).  (plan_decode_attn chooses the grid.)
//
// Each of the four consumer warps takes 16 of a stage's 64 slots.  A warp
// moves its K fragments into registers, runs QK^T, moves its V fragments
// into registers and frees the ring slot before the softmax and PV, so the
// slot refills while the warp computes.
template <int D, int NT, bool ON_READ, bool FUSE, bool KV8>
__global__ void __launch_bounds__(threads_of<FUSE>(), NT == 1 ? 2 : 1) attn_kernel(const __grid_constant__ AttnArgs args) {
  constexpr int KSTEPS = D / 16;  // k-steps of QK^T, m-tiles of PV
  constexpr int QSTR = D + 8;     // padded fp16 row stride of the query tiles
  constexpr int OSTR = D + 4;     // padded fp32 row stride of the output accumulator
  constexpr int ROWS = 8 * NT;
  constexpr int STAGE_ELEMS = kKS * D;
  constexpr int kStages = KV8 ? stages8_for<D>() : stages_for<D>();
  constexpr int STAGE_BYTES = KV8 ? stage8_bytes<D>() : 2 * STAGE_ELEMS * 2;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint16_t* kv_s = reinterpret_cast<uint16_t*>(smem);  // [stage][K | V][64][D] (fp8 store: bytes, + scales)
  // fp8 store: the expanded stage the consumers read, [K | V][64][D] 16-bit codes
  uint16_t* exp_s = reinterpret_cast<uint16_t*>(smem + kStages * STAGE_BYTES);
  uint16_t* qh_s = reinterpret_cast<uint16_t*>(smem + kStages * STAGE_BYTES + (KV8 ? 2 * STAGE_ELEMS * 2 : 0));  // [ROWS][QSTR] fp16 hi
  uint16_t* ql_s = qh_s + ROWS * QSTR;                 // [ROWS][QSTR] fp16 lo
  float* obuf = reinterpret_cast<float*>(ql_s + ROWS * QSTR);  // [2][ROWS][OSTR] fp32 partial sums
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ int new_done;  // fused append: units whose new rows the appender has written
  __shared__ float red_m[kCW][ROWS], red_l[kCW][ROWS];
  __shared__ float row_m[ROWS], row_l[ROWS];
  __shared__ int abort_flag, poisoned_s;
  __shared__ __align__(16) float lap_s[ON_READ ? D : 4];  // (cos, sin)(-C omega_i) of the unit's stream
  // the raw query of the next unit lands in shared memory (cp.async) on read, in registers otherwise
  constexpr bool STAGED = ON_READ && !FUSE;
  __shared__ __align__(16) uint16_t qraw_s[STAGED ? 8 * NT * D : 8];  // the unit's query rows as given

  const DevView& v = args.v;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = args.splits;
  const int hkv = v.n_kv_heads, hq = v.n_q_heads, group = hq / hkv, nq = v.q_per_step;
  const int rows = group * nq;
  const int n_active = args.n_active;
  const int n_units = n_active * hkv * args.n_layers;
  // this CTA's units: [u_first, n_units) with stride u_step; one unit when split
  const int split = splits > 1 ? static_cast<int>(blockIdx.x % splits) : 0;
  const int u_first = splits > 1 ? static_cast<int>(blockIdx.x / splits) : static_cast<int>(blockIdx.x);
  const int u_step = splits > 1 ? n_units : static_cast<int>(gridDim.x);

  // the producer's lanes touch every 32-byte line of the launch's parameters, so that the reads
  // after the dependency wait find them in the constant cache
  if (warp == kCW && lane * 32 < static_cast<int>(sizeof(AttnArgs))) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(&args)[lane * 8];
    asm volatile("" ::"r"(w));
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kCW);
    }
    new_done = 0;
    abort_flag = 0;
    // after a timed-out wait anywhere, later launches skip their copies (the
    // status word already reports the failure; each CTA ends quickly)
    poisoned_s = *reinterpret_cast<volatile int32_t*>(v.status) == DEV_TIMEOUT;
    asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const bool poisoned = poisoned_s != 0;

  if (warp == kCW) {
    // ---------------- producer: the warp walks every stage of every unit in the order the
    // consumers take them; lane 0 issues the bulk copies, the lanes hold 32 page-table
    // entries at a time, the next unit's descriptor is loaded a unit ahead.  With the append
    // fused, the copies of a stage that holds new tokens wait for the appender warp.
    if (!poisoned) {
      const int ps = v.page_size;
      const uint16_t* kreg = v.k_rot;
      const int copies = ps >= kKS ? 1 : kKS / ps;
      const int rows_per_copy = ps >= kKS ? kKS : ps;
      const uint32_t bytes = static_cast<uint32_t>(rows_per_copy) * D * (KV8 ? 1 : 2);
      int k = 0;  // stages walked so far (ring position)
      int k_issued = 0;  // stages walked up to the last one whose copies were issued
      bool stop = poisoned;
      int uj = 0;  // fused append: this CTA's units walked before the current one
      StepDesc dnext;
      int pbase = -64, pt_lane = 0;  // the lanes' 32-entry window of the unit's page-table row
      // the page table comes from rkv_create; the descriptors from the begin-step kernel, read
      // before the wait only when it ran two or more launches back (args.early), and then the
      // first unit's first page-table window with them; the pages may come from the immediate
      // predecessor: the bulk copies start after the wait
      const bool desc_early = (args.early & kEarlyDesc) != 0;
      if (u_first < n_units && desc_early && !stop) {
        dnext = v.desc[unit_of(u_first, n_active, hkv).a];
        pbase = split * args.stages_per_split * kKS / ps;
        pt_lane = pbase + lane < v.max_pages ? v.page_table[static_cast<int64_t>(dnext.stream) * v.max_pages + pbase + lane]
                                              : 0;
      }
      // the bulk copies of stage st of (layer, kv head) into ring buffer buf
      auto issue = [&](int st, int buf, int layer, int kvh, int stream_pages, const int32_t* ptab) {
        const uint32_t fb = smem_u32(&full_bar[buf]);
        if (lane == 0) mbar_arrive_expect_tx(fb, static_cast<uint32_t>(STAGE_BYTES));
        for (int c = 0; c < copies; ++c) {
          const int slot = st * kKS + c * rows_per_copy;
          int rp = slot / ps;
          const int off = slot % ps;
          if (rp >= stream_pages) rp = 0;  // past the window: any finite page (masked)
          if (rp < pbase || rp >= pbase + 32) {  // warp-uniform: refill the lanes' page-table window
            pbase = rp;
            pt_lane = pbase + lane < v.max_pages ? ptab[pbase + lane] : 0;
          }
          int page = __shfl_sync(0xffffffffu, pt_lane, rp - pbase);
          if (page < 0 || page >= v.n_pages) {
            if (lane == 0) record_error(v.status, DEV_BOUNDS, 21, page);
            page = 0;
          }
          if (lane == 0) {
            const int64_t src = pool_offset(v, layer, page, kvh, off);
            if constexpr (KV8) {  // fp8 keys, fp8 values (one byte per element) and the rows' scales
              const uint32_t dk = smem_u32(smem + buf * STAGE_BYTES + c * rows_per_copy * D);
              bulk_copy_g2s(dk, reinterpret_cast<const uint8_t*>(kreg) + src, bytes, fb);
              bulk_copy_g2s(dk + STAGE_ELEMS, reinterpret_cast<const uint8_t*>(v.v) + src, bytes, fb);
              bulk_copy_g2s(smem_u32(smem + buf * STAGE_BYTES + 2 * STAGE_ELEMS + c * rows_per_copy * 8),
                            v.kv_scale + src / D, static_cast<uint32_t>(rows_per_copy) * 8, fb);
            } else {
              const uint32_t dk = smem_u32(kv_s + buf * 2 * STAGE_ELEMS + c * rows_per_copy * D);
              bulk_copy_g2s(dk, kreg + src, bytes, fb);
              bulk_copy_g2s(dk + STAGE_ELEMS * 2, v.v + src, bytes, fb);
            }
          }
        }
      };
      // Fused append over keys that no launch of the step rewrites (offset-only, re-base applied
      // on read): the first unit's first stages hold none of the step's new rows (they are walked
      // last) and only pages that earlier steps wrote, so their copies start before the wait,
      // under the tail of the preceding launch.  A CTA with several units (its slot freed only as
      // the preceding launch's CTAs leave) takes a whole ring early; a CTA with one unit, which
      // may start while the preceding launch still streams, one stage (measured: a whole ring
      // there competes with that stream and costs more than it saves).
      int n_early = 0;
      const int early_cap = u_first + u_step < n_units ? kStages : 1;
      if (FUSE && u_first < n_units && desc_early && !stop && v.scheme != RKV_SCHEME_EXACT_REBASE &&
          v.withhold_stage < 0) {
        const Unit un = unit_of(u_first, n_active, hkv);
        const StepDesc& dsc = dnext;
        const int n_st = (slots_in_use(dsc) + kKS - 1) / kKS;
        const int st0 = split * args.stages_per_split;
        const int cnt = max(0, min(st0 + args.stages_per_split, n_st) - st0);
        const int first = first_new_slot(dsc);
        const int rot = walk_rot(first, v.q_per_step, dsc.ring, n_st);
        const int32_t* ptab = v.page_table + static_cast<int64_t>(dsc.stream) * v.max_pages;
        for (; n_early < early_cap && n_early < cnt; ++n_early) {
          const int st = st0 + n_early + rot >= n_st ? st0 + n_early + rot - n_st : st0 + n_early + rot;
          if (stage_has_new(first, v.q_per_step, dsc.ring, st)) break;
          issue(st, n_early, args.layer0 + un.lz, un.kvh, (dsc.ring + ps - 1) / ps, ptab);
        }
        k = k_issued = n_early;
      }
      pdl_wait();
      pdl_launch_dependents();
      if (u_first < n_units && !(desc_early && !poisoned)) dnext = v.desc[unit_of(u_first, n_active, hkv).a];
      for (int u = u_first; u < n_units; u += u_step, ++uj) {
        const Unit un = unit_of(u, n_active, hkv);
        const StepDesc dsc = dnext;
        if (u + u_step < n_units) dnext = v.desc[unit_of(u + u_step, n_active, hkv).a];  // lands during this unit
        const int layer = args.layer0 + un.lz;
        const int n_st = (slots_in_use(dsc) + kKS - 1) / kKS;
        const int st0 = split * args.stages_per_split;
        const int cnt = max(0, min(st0 + args.stages_per_split, n_st) - st0);
        const int first = FUSE ? first_new_slot(dsc) : 0;
        const int rot = FUSE ? walk_rot(first, v.q_per_step, dsc.ring, n_st) : 0;
        const int stream_pages = (dsc.ring + ps - 1) / ps;
        const int32_t* ptab = v.page_table + static_cast<int64_t>(dsc.stream) * v.max_pages;
        if (u != u_first) pbase = -64;  // another stream's row
        for (int i = u == u_first ? n_early : 0; i < cnt; ++i, ++k) {
          const int st = FUSE && st0 + i + rot >= n_st ? st0 + i + rot - n_st : st0 + i + rot;
          const int buf = k % kStages;
          if (!stop && k >= kStages &&
              !__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[buf]), ((k / kStages) - 1) & 1, v.wait_ns))) {
            if (lane == 0) {
              record_error(v.status, DEV_TIMEOUT, 20, k);
              atomicExch(&abort_flag, 1);
            }
            stop = true;
          }
          if (!stop && __any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&abort_flag) != 0)) stop = true;
          // fused append: a stage with new tokens is copied once the appender has written the
          // unit's rows into the pool
          if (FUSE && !stop && stage_has_new(first, v.q_per_step, dsc.ring, st) &&
              !__all_sync(0xffffffffu, wait_count(&new_done, uj + 1, v.wait_ns))) {
            if (lane == 0) {
              record_error(v.status, DEV_TIMEOUT, 25, k);
              atomicExch(&abort_flag, 1);
            }
            stop = true;
          }
          if (!stop) k_issued = k + 1;
          // the failure-detection test hook: this stage's copy never starts, so its consumers'
          // bounded wait runs out
          if (stop || k == v.withhold_stage) continue;
          issue(st, buf, layer, un.kvh, stream_pages, ptab);
        }
      }
      // never leave with copies in flight (only reachable on an aborted run): the last kStages
      // stages whose copies were issued
      if (lane == 0)
        for (int i = max(0, k_issued - kStages); i < k_issued; ++i)
          if (i != v.withhold_stage && !mbar_wait(smem_u32(&full_bar[i % kStages]), (i / kStages) & 1, v.wait_ns))
            record_error(v.status, DEV_TIMEOUT, 22, i);
    }
  } else if (FUSE && warp == kCW + 1) {
    // ---------------- appender (fused append): after the wait, since the new keys and values may
    // come from the immediate predecessor, the new tokens of every unit the CTA walks that fall in
    // its stages, publishing the count of units done after each.  It runs in a launch that skips
    // its copies too.
    pdl_wait();
    int done = 0;
    for (int u = u_first; u < n_units; u += u_step) {
      const Unit un = unit_of(u, n_active, hkv);
      const StepDesc dsc = v.desc[un.a];
      const int n_st = (slots_in_use(dsc) + kKS - 1) / kKS;
      const int first = first_new_slot(dsc);
      const int rot = walk_rot(first, nq, dsc.ring, n_st);
      const int st0 = split * args.stages_per_split;
      for (int t = 0; t < nq && n_st > 0; ++t) {
        const int slot = new_slot(first, t, dsc.ring);
        const int i = (slot / kKS - rot + n_st) % n_st;
        if (i >= st0 && i < st0 + args.stages_per_split) {
          if constexpr (KV8)
            append_token_e4m3<D>(args, dsc, un, t, slot, lane);
          else
            append_token<D>(args, dsc, un, t, slot, lane);
        }
      }
      fence_proxy_async_global();  // the rows precede the producer's bulk copies
      __syncwarp();
      if (lane == 0) st_release_smem(&new_done, ++done);
    }
  } else if (!poisoned) {
    // ---------------- consumers
    const int tid = threadIdx.x;
    const int wt = warp;  // this warp's 16 slots of each stage: wt*16 .. wt*16+15
    const int g = lane >> 2, tq = lane & 3;
    // ldmatrix lane roles: matrix mi = lane / 8, row ri = lane % 8
    const int mi = lane >> 3, ri = lane & 7;
    const int krow = wt * 16 + ri + (mi & 1) * 8, kchunk = mi >> 1;  // K as the A operand
    const int vrow = wt * 16 + ri + (mi >> 1) * 8, vchunk = mi & 1;  // V^T as the A operand
    QPrefetch<D> pf;
    StepDesc dnext;
    // descriptors, angles and queries before the wait only as args.early allows
    const bool desc_early = (args.early & kEarlyDesc) != 0, q_early = (args.early & kEarlyQ) != 0;
    if (u_first < n_units) {
      const Unit un0 = unit_of(u_first, n_active, hkv);
      if (desc_early) dnext = v.desc[un0.a];
      if (desc_early && q_early) q_prefetch<D, STAGED>(args, un0, tid, pf, qraw_s, ON_READ ? lap_s : nullptr);
    }
    pdl_wait();
    if (u_first < n_units) {
      const Unit un0 = unit_of(u_first, n_active, hkv);
      if (!desc_early) dnext = v.desc[un0.a];
      if (!(desc_early && q_early)) q_prefetch<D, STAGED>(args, un0, tid, pf, qraw_s, ON_READ ? lap_s : nullptr);
    }
    int k0 = 0;  // ring position of the unit's first stage
    for (int u = u_first; u < n_units; u += u_step) {
      const Unit un = unit_of(u, n_active, hkv);
      const StepDesc dsc = dnext;
      const int W = dsc.ring, len = dsc.len;  // W: the ring's modulus
      const int nslots = slots_in_use(dsc);
      const int n_st = (nslots + kKS - 1) / kKS;
      const int st0 = split * args.stages_per_split;
      const int my_st = max(0, min(st0 + args.stages_per_split, n_st) - st0);
      // fused append: the slot of the walk's current stage, from stage rot + st0 on, wrapping
      int sb = 0;
      if (FUSE) {
        const int st = walk_rot(first_new_slot(dsc), nq, dsc.ring, n_st) + st0;
        sb = (st >= n_st ? st - n_st : st) * kKS;
      }

      if constexpr (STAGED) cp_async_wait_all();  // own raw query chunks, lap element (S1 publishes it)
      q_build<D, NT, STAGED>(pf, v.scale_log2, tid, qh_s, ql_s, qraw_s, rows);
      if constexpr (ON_READ && !STAGED) {
        if (tid < D) lap_s[tid] = pf.lap;
      }
      consumer_sync();  // S1: query tiles ready; the previous unit's output pass is over
      // on read: the next lap's query tiles (R(-C) applied), for the ring slots below evicted mod
      // C, in the output tiles' space (free until this unit's epilogue)
      uint16_t* const nh_s = reinterpret_cast<uint16_t*>(obuf);
      uint16_t* const nl_s = nh_s + ROWS * QSTR;
      if constexpr (ON_READ) {
        if (dsc.evicted % W != 0) {  // uniform: some retained tokens are on the next lap
          build_next_lap<D, NT>(qh_s, ql_s, nh_s, nl_s, lap_s, tid);
          consumer_sync();  // S1b
        }
      }
      uint32_t qh[NT][KSTEPS][2], ql[NT][KSTEPS][2];
      auto load_q = [&](const uint16_t* th, const uint16_t* tl) {  // query fragments (B operand)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const int base = (nt * 8 + g) * QSTR + ks * 16 + 2 * tq;
            qh[nt][ks][0] = *reinterpret_cast<const uint32_t*>(th + base);
            qh[nt][ks][1] = *reinterpret_cast<const uint32_t*>(th + base + 8);
            if constexpr (!KV8) {
              ql[nt][ks][0] = *reinterpret_cast<const uint32_t*>(tl + base);
              ql[nt][ks][1] = *reinterpret_cast<const uint32_t*>(tl + base + 8);
            }
          }
      };
      load_q(qh_s, ql_s);
      // on read: whether the fragments hold the next lap's query
      bool lap_b = false;
      if (u + u_step < n_units) {  // the next unit's query and descriptor land during this unit
        const Unit un1 = unit_of(u + u_step, n_active, hkv);
        // lap_s is free: this unit's next-lap tile is built (S1b), or was not needed
        q_prefetch<D, STAGED>(args, un1, tid, pf, qraw_s, ON_READ ? lap_s : nullptr);
        dnext = v.desc[un1.a];
      }

      float m_run[NT][2], l_run[NT][2], o_acc[KSTEPS][NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
        l_run[nt][0] = l_run[nt][1] = 0.f;
      }
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o_acc[mt][nt][e] = 0.f;

      const int ev_mod = static_cast<int>(dsc.evicted % W);
      const int first_new = len - nq;  // window index of the step's first new token
      bool aborted = false;
      for (int i = 0; i < my_st; ++i, sb = sb + kKS >= nslots ? 0 : sb + kKS) {
        const int k = k0 + i;
        const int buf = k % kStages;
        // warp-uniform decision: every lane leaves together if any lane gave up
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[buf]), (k / kStages) & 1, v.wait_ns))) {
          if (lane == 0) {
            record_error(v.status, DEV_TIMEOUT, 23, k);
            atomicExch(&abort_flag, 1);
          }
          aborted = true;
          break;
        }
        const int slot_base = (FUSE ? sb : (st0 + i) * kKS) + wt * 16;
        const uint32_t kb = smem_u32(KV8 ? exp_s : kv_s + buf * 2 * STAGE_ELEMS);
        const uint32_t vb = kb + STAGE_ELEMS * 2;
        if (slot_base >= nslots) {  // none of this warp's slots holds a token
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty_bar[buf]));
          continue;
        }
        // fp8 store: the warp expands its 16 rows into the 16-bit stage (two lanes a row): key codes
        // as fp16 (exact), values as fp16 code * 2^e (exact unless a row's scale is below 2^-15,
        // where the smallest codes lose bits below 2^-24), takes its two keys' scales and frees the
        // ring slot at once.  Scores are scaled by the key's 2^e; the values then need an fp16
        // product with the softmax weights.
        float sk[2] = {1.f, 1.f};
        if constexpr (KV8) {
          const uint8_t* st8 = smem + buf * STAGE_BYTES;
          constexpr int C8 = D / 16;       // 16-byte chunks of codes per row
          constexpr int RPP = 32 / C8;     // rows per pass: C8 lanes read a row's codes side by side
          const int c = lane % C8;         // codes 16c .. 16c + 15 = 16-bit chunks 2c, 2c + 1
          __syncwarp();  // the previous stage's fragment loads of these rows are done
#pragma unroll 1
          for (int j = 0; j < 16 / RPP; ++j) {  // one pass at a time: the consumers sit at the register limit
            const int r = wt * 16 + j * RPP + lane / C8;
            const __half2 vs2 = __float2half2_rn(reinterpret_cast<const float2*>(st8 + 2 * STAGE_ELEMS)[r].y);
            const uint32_t vsc = *reinterpret_cast<const uint32_t*>(&vs2);
            auto vscale = [&](uint32_t h2) {  // fp16x2 codes times the row's value scale
              uint32_t y;
              asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(h2), "r"(vsc));
              return y;
            };
            const uint4 kq = *reinterpret_cast<const uint4*>(st8 + r * D + c * 16);
            const uint4 vq = *reinterpret_cast<const uint4*>(st8 + STAGE_ELEMS + r * D + c * 16);
            const uint4 k0 = make_uint4(e4m3x2_to_f16x2(kq.x & 0xFFFFu), e4m3x2_to_f16x2(kq.x >> 16),
                                        e4m3x2_to_f16x2(kq.y & 0xFFFFu), e4m3x2_to_f16x2(kq.y >> 16));
            const uint4 k1 = make_uint4(e4m3x2_to_f16x2(kq.z & 0xFFFFu), e4m3x2_to_f16x2(kq.z >> 16),
                                        e4m3x2_to_f16x2(kq.w & 0xFFFFu), e4m3x2_to_f16x2(kq.w >> 16));
            const uint4 v0 = make_uint4(vscale(e4m3x2_to_f16x2(vq.x & 0xFFFFu)), vscale(e4m3x2_to_f16x2(vq.x >> 16)),
                                        vscale(e4m3x2_to_f16x2(vq.y & 0xFFFFu)), vscale(e4m3x2_to_f16x2(vq.y >> 16)));
            const uint4 v1 = make_uint4(vscale(e4m3x2_to_f16x2(vq.z & 0xFFFFu)), vscale(e4m3x2_to_f16x2(vq.z >> 16)),
                                        vscale(e4m3x2_to_f16x2(vq.w & 0xFFFFu)), vscale(e4m3x2_to_f16x2(vq.w >> 16)));
            *reinterpret_cast<uint4*>(exp_s + r * D + swizzle_chunk(2 * c, r) * 8) = k0;
            *reinterpret_cast<uint4*>(exp_s + r * D + swizzle_chunk(2 * c + 1, r) * 8) = k1;
            *reinterpret_cast<uint4*>(exp_s + STAGE_ELEMS + r * D + swizzle_chunk(2 * c, r) * 8) = v0;
            *reinterpret_cast<uint4*>(exp_s + STAGE_ELEMS + r * D + swizzle_chunk(2 * c + 1, r) * 8) = v1;
          }
          const float2* sc = reinterpret_cast<const float2*>(st8 + 2 * STAGE_ELEMS);
          sk[0] = sc[wt * 16 + g].x;
          sk[1] = sc[wt * 16 + g + 8].x;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty_bar[buf]));
        }
        // window index (token - evicted) of this thread's two keys; -1 = empty slot
        int widx[2];
#pragma unroll
        for (int hk = 0; hk < 2; ++hk) {
          const int slot = slot_base + g + 8 * hk;
          int w = slot - ev_mod;
          if (w < 0) w += W;
          widx[hk] = slot < nslots ? w : -1;
        }
        // K fragments of this warp's 16 slots (the A operand, one per k-step)
        uint32_t kf[KSTEPS][4];
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) ldsm_x4(kb + krow * D * 2 + (swizzle_chunk(2 * ks + kchunk, ri) << 4), kf[ks]);
        float sh[NT][4], sl[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sh[nt][e] = sl[nt][e] = 0.f;
        auto qk = [&](float (&ah)[NT][4], float (&al)[NT][4]) {
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_f16(ah[nt], kf[ks], qh[nt][ks][0], qh[nt][ks][1]);
              // the query's low part: fp32 accuracy against fp16 keys; the fp8 store's keys carry
              // 2^-4 relative error, where the fp16 query alone (2^-11) is already far below it
              if constexpr (!KV8) mma_f16(al[nt], kf[ks], ql[nt][ks][0], ql[nt][ks][1]);
            }
        };
        if constexpr (ON_READ) {
          // warp-uniform: slots [slot_base, slot_base + 16) against ev_mod
          if (slot_base + 16 <= ev_mod) {         // all of the next lap
            if (!lap_b) load_q(nh_s, nl_s);
            lap_b = true;
            qk(sh, sl);
          } else if (slot_base >= ev_mod) {       // all of the current lap
            if (lap_b) load_q(qh_s, ql_s);
            lap_b = false;
            qk(sh, sl);
          } else {                                // the chunk where the two laps meet
            float bh[NT][4], bl[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) bh[nt][e] = bl[nt][e] = 0.f;
            if (!lap_b) load_q(nh_s, nl_s);
            qk(bh, bl);
            load_q(qh_s, ql_s);
            lap_b = false;
            qk(sh, sl);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (slot_base + g + 8 * (e >> 1) < ev_mod) {
                  sh[nt][e] = bh[nt][e];
                  sl[nt][e] = bl[nt][e];
                }
          }
        } else {
          qk(sh, sl);
        }
        // V fragments (V^T as the A operand, one per m-tile), then the slot refills while we compute
        uint32_t vf[KSTEPS][4];
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) ldsm_x4_t(vb + vrow * D * 2 + (swizzle_chunk(2 * mt + vchunk, ri) << 4), vf[mt]);
        if constexpr (!KV8) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty_bar[buf]));
        }
        // online softmax; C layout: e = 0,1 key g rows 2tq, 2tq+1; e = 2,3 key g+8.  A chunk
        // whose slots all hold tokens that every query of the step sees needs no mask (one query
        // and every written slot in the window: no test needed).
        const bool full_chunk = slot_base + 16 <= nslots &&
                                ((nq == 1 && len == nslots) ||
                                 __all_sync(0xffffffffu, widx[0] <= first_new && widx[1] <= first_new));
        uint32_t pb[NT][2];
        float alpha[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float s[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int wi = widx[e >> 1];
            const int row = nt * 8 + 2 * tq + (e & 1);
            // causal inside the step: query t sees window index <= first_new + t
            const bool ok = full_chunk || (wi >= 0 && wi <= first_new + min(row / group, nq - 1));
            s[e] = ok ? (sh[nt][e] + sl[nt][e]) * sk[e >> 1] : -CUDART_INF_F;
          }
          float p[4];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float mx = fmaxf(s[c], s[c + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[nt][c], mx);
            const float base = m_new == -CUDART_INF_F ? 0.f : m_new;
            alpha[nt][c] = fast_exp2(m_run[nt][c] - base);
            p[c] = fast_exp2(s[c] - base);
            p[c + 2] = fast_exp2(s[c + 2] - base);
            l_run[nt][c] = l_run[nt][c] * alpha[nt][c] + p[c] + p[c + 2];
            m_run[nt][c] = m_new;
          }
          if constexpr (KV8) {  // fp16 weights against the fp16 values
            pb[nt][0] = movmatrix_t(pack_f16(p[0], p[1]));
            pb[nt][1] = movmatrix_t(pack_f16(p[2], p[3]));
          } else {
            pb[nt][0] = movmatrix_t(pack_bf16(p[0], p[1]));
            pb[nt][1] = movmatrix_t(pack_bf16(p[2], p[3]));
          }
        }
        // rescale the accumulators only when some row's running max moved in this warp
        bool moved = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) moved = moved || alpha[nt][0] != 1.f || alpha[nt][1] != 1.f;
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              o_acc[mt][nt][0] *= alpha[nt][0];
              o_acc[mt][nt][1] *= alpha[nt][1];
              o_acc[mt][nt][2] *= alpha[nt][0];
              o_acc[mt][nt][3] *= alpha[nt][1];
            }
        }
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if constexpr (KV8)
              mma_f16(o_acc[mt][nt], vf[mt], pb[nt][0], pb[nt][1]);
            else
              mma_bf16(o_acc[mt][nt], vf[mt], pb[nt][0], pb[nt][1]);
          }
      }
      k0 += my_st;

      // ---------------- combine the warps: rescale in registers, add in shared memory
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float l = l_run[nt][c];
          l += __shfl_xor_sync(0xffffffffu, l, 4);
          l += __shfl_xor_sync(0xffffffffu, l, 8);
          l += __shfl_xor_sync(0xffffffffu, l, 16);
          l_run[nt][c] = l;
          if (g == 0) {
            red_m[warp][nt * 8 + 2 * tq + c] = m_run[nt][c];
            red_l[warp][nt * 8 + 2 * tq + c] = l;
          }
        }
      consumer_sync();  // S2
      float sc[NT][2];  // this warp's rescale factor per row
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int row = nt * 8 + 2 * tq + c;
          float mx = -CUDART_INF_F;
#pragma unroll
          for (int w = 0; w < kCW; ++w) mx = fmaxf(mx, red_m[w][row]);
          const float f = m_run[nt][c] == -CUDART_INF_F ? 0.f : exp2f(m_run[nt][c] - mx);
          if (warp == 0 && g == 0) {
            float lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w)
              if (red_m[w][row] != -CUDART_INF_F) lsum += red_l[w][row] * exp2f(red_m[w][row] - mx);
            row_m[row] = mx;
            row_l[row] = lsum;
          }
          // deterministic sum: warps 0, 1 store into tiles 0, 1, then warps 2, 3 add theirs
          if (warp < 2) {
            float* tile = obuf + warp * ROWS * OSTR + row * OSTR;
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
              tile[mt * 16 + g] = o_acc[mt][nt][c] * f;
              tile[mt * 16 + g + 8] = o_acc[mt][nt][c + 2] * f;
            }
          }
          sc[nt][c] = f;
        }
      consumer_sync();  // S2b: tiles 0 and 1 hold warps 0 and 1
      if (warp >= 2) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float* tile = obuf + (warp - 2) * ROWS * OSTR + (nt * 8 + 2 * tq + c) * OSTR;
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) {
              tile[mt * 16 + g] += o_acc[mt][nt][c] * sc[nt][c];
              tile[mt * 16 + g + 8] += o_acc[mt][nt][c + 2] * sc[nt][c];
            }
          }
      }
      // S3: tiles 0 + 1 hold the CTA's unnormalised output, row_m / row_l its statistics; a wait that
      // gave up in any warp ends the unit loop for all of them
      if (consumer_sync_or(aborted)) break;

      if (args.mode == 1) break;  // the cluster combine below finishes this (single) unit
      // ---------------- output pass: thread -> (row, 8 consecutive dims)
      constexpr int CH = D / 8;
      for (int e = tid; e < rows * CH; e += kCW * 32) {
        const int row = e / CH, ch = e % CH;
        const float* src = obuf + row * OSTR + ch * 8;
        const float4 a0 = *reinterpret_cast<const float4*>(src), a1 = *reinterpret_cast<const float4*>(src + 4);
        const float4 b0 = *reinterpret_cast<const float4*>(src + ROWS * OSTR);
        const float4 b1 = *reinterpret_cast<const float4*>(src + ROWS * OSTR + 4);
        const float4 o0 = make_float4(a0.x + b0.x, a0.y + b0.y, a0.z + b0.z, a0.w + b0.w);
        const float4 o1 = make_float4(a1.x + b1.x, a1.y + b1.y, a1.z + b1.z, a1.w + b1.w);
        const float mx = row_m[row], lsum = row_l[row];
        const int t = row / group, h = un.kvh * group + row % group;
        const int64_t orow = (static_cast<int64_t>(un.a) * nq + t) * hq + h;
        if (args.mode == 0) {
          const float inv = 1.f / lsum;
          const float o[8] = {o0.x * inv, o0.y * inv, o0.z * inv, o0.w * inv,
                              o1.x * inv, o1.y * inv, o1.z * inv, o1.w * inv};
          *reinterpret_cast<uint4*>(args.out + un.lz * args.q_layer_stride + orow * D + ch * 8) = pack8_bf16(o);
          if (args.lse && ch == 0)
            args.lse[un.lz * args.lse_layer_stride + orow] = (mx + log2f(lsum)) * 0.69314718055994531f;
        } else {  // mode 2: normalised partials of this split
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          const int64_t prow = orow * splits + split;
          float4* dst = reinterpret_cast<float4*>(v.part_o + prow * D + ch * 8);
          dst[0] = make_float4(o0.x * inv, o0.y * inv, o0.z * inv, o0.w * inv);
          dst[1] = make_float4(o1.x * inv, o1.y * inv, o1.z * inv, o1.w * inv);
          if (ch == 0) {
            v.part_ml[prow * 2] = mx;
            v.part_ml[prow * 2 + 1] = lsum;
          }
        }
      }
    }
    // a unit loop left early (a wait gave up) may leave the next unit's staged copies in flight
    if constexpr (STAGED) cp_async_wait_all();
  }

  if (args.mode == 1) {
    // ---------------- combine the cluster's splits through distributed shared memory
    __syncwarp();
    cluster_sync_all();
    const uint32_t rank = cluster_rank();
    if (warp < kCW && !poisoned) {
      const Unit un = unit_of(u_first, n_active, hkv);
      constexpr int CH = D / 8;
      for (int e = static_cast<int>(rank) * kCW * 32 + threadIdx.x; e < rows * CH; e += splits * kCW * 32) {
        const int row = e / CH, ch = e % CH;
        float mr[8], lr[8];
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r < splits) {
            mr[r] = ld_dsmem_f32(&row_m[row], r);
            lr[r] = ld_dsmem_f32(&row_l[row], r);
          } else {
            mr[r] = -CUDART_INF_F;
            lr[r] = 0.f;
          }
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) mx = fmaxf(mx, mr[r]);
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float lsum = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r < splits && mr[r] != -CUDART_INF_F) {
            const float f = exp2f(mr[r] - mx);
            const float4 t0 = ld_dsmem_f32x4(obuf + row * OSTR + ch * 8, r);
            const float4 t1 = ld_dsmem_f32x4(obuf + row * OSTR + ch * 8 + 4, r);
            const float4 u0 = ld_dsmem_f32x4(obuf + ROWS * OSTR + row * OSTR + ch * 8, r);
            const float4 u1 = ld_dsmem_f32x4(obuf + ROWS * OSTR + row * OSTR + ch * 8 + 4, r);
            const float4 a0 = make_float4(t0.x + u0.x, t0.y + u0.y, t0.z + u0.z, t0.w + u0.w);
            const float4 a1 = make_float4(t1.x + u1.x, t1.y + u1.y, t1.z + u1.z, t1.w + u1.w);
            lsum += lr[r] * f;
            o[0] += a0.x * f;
            o[1] += a0.y * f;
            o[2] += a0.z * f;
            o[3] += a0.w * f;
            o[4] += a1.x * f;
            o[5] += a1.y * f;
            o[6] += a1.z * f;
            o[7] += a1.w * f;
          }
        }
        const float inv = 1.f / lsum;
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] *= inv;
        const int t = row / group, h = un.kvh * group + row % group;
        const int64_t orow = (static_cast<int64_t>(un.a) * nq + t) * hq + h;
        *reinterpret_cast<uint4*>(args.out + un.lz * args.q_layer_stride + orow * D + ch * 8) = pack8_bf16(o);
        if (args.lse && ch == 0) args.lse[un.lz * args.lse_layer_stride + orow] = (mx + log2f(lsum)) * 0.69314718055994531f;
      }
    }
    cluster_sync_all();  // keep this CTA's shared memory alive until every rank has read it
  }
}

// One block per (active stream, query row): combine the splits' partials.
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(DevView v, int splits, uint16_t* __restrict__ out,
                                                    float* __restrict__ lse) {
  pdl_wait();
  pdl_launch_dependents();
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

template <int D, int NT, bool ON_READ, bool FUSE, bool KV8>
struct Kernel {
  static constexpr int kSmem = smem_bytes_for<D, NT, KV8>();
  // The dynamic shared-memory opt-in is per device, so it and the occupancy it gives are
  // set up once for every device the process uses.
  static int occupancy() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int occ[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (occ[dev] == 0) {
      cudaFuncSetAttribute(attn_kernel<D, NT, ON_READ, FUSE, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      int o = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, attn_kernel<D, NT, ON_READ, FUSE, KV8>, threads_of<FUSE>(),
                                                        kSmem) != cudaSuccess)
        o = 1;
      occ[dev] = o < 1 ? 1 : o;
    }
    return occ[dev];
  }
  static cudaError_t launch(const AttnArgs& args, int grid, cudaStream_t st) {
    occupancy();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads_of<FUSE>());
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (args.mode == 1) {
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = args.splits;
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, attn_kernel<D, NT, ON_READ, FUSE, KV8>, args);
  }
};

template <int D, int NT>
int occupancy_of(bool on_read, bool kv8) {
  if constexpr (NT == 1) {
    if (kv8) return on_read ? Kernel<D, 1, true, false, true>::occupancy() : Kernel<D, 1, false, false, true>::occupancy();
  }
  return on_read ? Kernel<D, NT, true, false, false>::occupancy() : Kernel<D, NT, false, false, false>::occupancy();
}

int occupancy_for(const DevView& v) {
  const bool two = v.n_q_heads / v.n_kv_heads * v.q_per_step > 8;
  const bool on_read = v.scheme == RKV_SCHEME_EXACT_ON_READ, kv8 = v.kv_scale != nullptr;
  if (v.head_dim == 128) return two ? occupancy_of<128, 2>(on_read, kv8) : occupancy_of<128, 1>(on_read, kv8);
  return two ? occupancy_of<64, 2>(on_read, kv8) : occupancy_of<64, 1>(on_read, kv8);
}

template <int D, int NT, bool KV8>
cudaError_t dispatch_fused(const AttnArgs& args, int grid, cudaStream_t st) {
  const bool fuse = args.k_new != nullptr;
  if (args.v.scheme == RKV_SCHEME_EXACT_ON_READ)
    return fuse ? Kernel<D, NT, true, true, KV8>::launch(args, grid, st)
                : Kernel<D, NT, true, false, KV8>::launch(args, grid, st);
  return fuse ? Kernel<D, NT, false, true, KV8>::launch(args, grid, st)
              : Kernel<D, NT, false, false, KV8>::launch(args, grid, st);
}

template <int D, int NT>
cudaError_t dispatch_on_read(const AttnArgs& args, int grid, cudaStream_t st) {
  if constexpr (NT == 1) {
    if (args.v.kv_scale) return dispatch_fused<D, 1, true>(args, grid, st);
  } else {
    if (args.v.kv_scale) return cudaErrorInvalidValue;  // the fp8 store takes up to 8 query rows a kv head
  }
  return dispatch_fused<D, NT, false>(args, grid, st);
}

cudaError_t dispatch(const AttnArgs& args, int grid, cudaStream_t st) {
  const DevView& v = args.v;
  const bool two = v.n_q_heads / v.n_kv_heads * v.q_per_step > 8;
  if (v.head_dim == 128) return two ? dispatch_on_read<128, 2>(args, grid, st) : dispatch_on_read<128, 1>(args, grid, st);
  return two ? dispatch_on_read<64, 2>(args, grid, st) : dispatch_on_read<64, 1>(args, grid, st);
}

int64_t resident_ctas(const DevView& v) {
  return static_cast<int64_t>(v.num_sms > 0 ? v.num_sms : 148) * occupancy_for(v);
}

AttnArgs make_args(const DevView& v, int n_active, int layer0, int n_layers, const uint16_t* q, uint16_t* out,
                   float* lse, int64_t q_layer_stride, int64_t lse_layer_stride, const AttnPlan& p) {
  AttnArgs args;
  args.v = v;
  args.q = q;
  args.out = out;
  args.lse = lse;
  args.q_layer_stride = q_layer_stride;
  args.lse_layer_stride = lse_layer_stride;
  args.layer0 = layer0;
  args.n_layers = n_layers;
  args.n_active = n_active;
  args.splits = p.splits;
  args.stages_per_split = p.stages_per_split;
  args.mode = 0;
  args.early = 0;
  args.k_new = nullptr;
  args.v_new = nullptr;
  args.kv_layer_stride = 0;
  return args;
}

}  // namespace

AttnPlan plan_decode_attn(const DevView& v, int n_active, int n_layers, bool cluster) {
  // the page table bounds every stream's window by max_pages * page_size
  const int max_stages = (v.max_pages * v.page_size + kKS - 1) / kKS;
  const int64_t units = static_cast<int64_t>(n_active) * v.n_kv_heads * n_layers;
  const int64_t sms = v.num_sms > 0 ? v.num_sms : 148;
  const int ring = v.head_dim == 128 ? stages_for<128>() : stages_for<64>();
  // One layer of few, short windows: at most one CTA per SM, so that the next launch's CTAs
  // find a free slot, start as soon as this launch lets them (programmatic dependent launch)
  // and hold their descriptors and queries when it completes.  Long windows or many units
  // keep every CTA slot streaming.
  const bool one_per_sm = n_layers == 1 && units <= sms && max_stages <= 4 * ring;
  const int64_t slots = one_per_sm ? sms : resident_ctas(v);
  int splits = 1;
  // fewer units than CTA slots: split every window over several CTAs
  if (units < slots) splits = static_cast<int>(slots / units);
  const int cap = cluster ? 8 : 64;
  splits = splits > cap ? cap : splits;
  splits = splits > max_stages ? max_stages : splits;
  splits = splits < 1 ? 1 : splits;
  const int sps = (max_stages + splits - 1) / splits;
  splits = (max_stages + sps - 1) / sps;
  AttnPlan p;
  p.splits = splits;
  p.stages_per_split = splits > 1 ? sps : max_stages;
  p.cluster = cluster && splits > 1;
  p.slots = slots;
  return p;
}

cudaError_t launch_decode_attn(const DevView& v, int n_active, int layer0, int n_layers, const uint16_t* q,
                               uint16_t* out, float* lse, int64_t q_layer_stride, int64_t lse_layer_stride,
                               const AttnExtras& x, cudaStream_t st) {
  const AttnPlan p = plan_decode_attn(v, n_active, n_layers, true);
  AttnArgs args = make_args(v, n_active, layer0, n_layers, q, out, lse, q_layer_stride, lse_layer_stride, p);
  args.early = x.early;
  args.k_new = x.k_new;
  args.v_new = x.v_new;
  args.kv_layer_stride = x.kv_layer_stride;
  const int64_t units = static_cast<int64_t>(n_active) * v.n_kv_heads * n_layers;
  args.mode = p.cluster ? 1 : 0;
  const int64_t grid = p.cluster ? units * p.splits : (units < p.slots ? units : p.slots);
  return dispatch(args, static_cast<int>(grid), st);
}

cudaError_t launch_decode_attn_scratch(const DevView& v, int n_active, int layer, const uint16_t* q, uint16_t* out,
                                       float* lse, cudaStream_t st) {
  const AttnPlan p = plan_decode_attn(v, n_active, 1, false);
  AttnArgs args = make_args(v, n_active, layer, 1, q, out, lse, 0, 0, p);
  const int64_t units = static_cast<int64_t>(n_active) * v.n_kv_heads;
  args.mode = p.splits > 1 ? 2 : 0;
  args.early = kEarlyDesc;  // rkv_append_rope ran after the begin-step kernel
  const int64_t grid = p.splits > 1 ? units * p.splits : (units < p.slots ? units : p.slots);
  cudaError_t e = dispatch(args, static_cast<int>(grid), st);
  if (e != cudaSuccess || p.splits == 1) return e;
  const int blocks = n_active * v.q_per_step * v.n_q_heads;
  if (v.head_dim == 128) return launch_pdl(merge_kernel<128>, dim3(blocks), dim3(128), 0, st, v, p.splits, out, lse);
  return launch_pdl(merge_kernel<64>, dim3(blocks), dim3(64), 0, st, v, p.splits, out, lse);
}

}  // namespace rkv

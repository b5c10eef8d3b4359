// m3scan.cu -- selective-scan layer core (Mamba-1), forward and backward, for
// sm_103a.  The C ABI is declared in include/m3scan.h.
//
// What is computed follows the mamba-rs pages: src/mamba_ssm/gpu/
// forward_mixed.rs (0.3.1), steps F4a conv1d + SiLU, F4c softplus, F4d the
// selective scan with the D skip, F4e gating, and the backward scratch list
// of the same page; A = -exp(a_log) from trainer.rs (0.7.3),
// recompute_a_neg_all.  The design is not the pages': they save the f32
// state before every step (h_saved, B*(T+1)*d_inner*d_state) and the
// discretisation da_exp per step.  Here the forward keeps the 16 state lanes
// of one channel in registers and writes only the state at the start of each
// chunk of K steps; the backward recomputes one chunk at a time into shared
// memory and runs the reverse-time pass from there.
//
// Work decomposition.  A block owns (batch b, a group of 64 channels, one
// time segment); a thread owns one channel and all 16 lanes of its state.
// When batch * channel groups alone cannot fill the GPU, time is split into
// S segments of whole chunks.  The scan is linear in the state, so a
// segment's effect on the next one is (decay, local end state): an
// aggregate kernel computes it per segment, a carry kernel chains the
// segments, and the main kernel reruns each segment from its true start.
// The backward does the same in reverse time for the adjoint state.
//
// dB and dC are sums over channels: each warp reduces its 32 channels with
// a shuffle reduce-scatter, warps combine in shared memory, and each block
// adds one float per (t, n) to the f32 output with a global reduction.
// Parameter gradients are written as per-(batch, segment) partials and
// summed in a fixed order by a finalize kernel (deterministic).

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "../../include/m3scan.h"

// Backward scratch owned by the library itself, for m3scan_bwd_noalloc.
// Every GPU that loads this library holds these bytes until the process
// exits.  Host code must not use the name as an address: it is fetched per
// device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[M3SCAN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int NS = 16;        // d_state lanes per channel
constexpr int WC = 4;         // conv taps
constexpr int GF = 128;       // forward: channels (= threads) per block
constexpr int GB = 128;       // backward: channels (= threads) per block = 4 warps,
                              // one per tensor-memory lane quadrant
constexpr int NWB = GB / 32;  // backward warps per block
constexpr int TT = 16;        // forward / aggregate staging tile (steps)
constexpr int SUB = 8;        // forward scalar sub-tile (steps)
constexpr int KMAX = 64;      // largest chunk (the backward may allow less)
constexpr int KDEF = 8;       // default chunk
constexpr int NPART = 24;     // per-channel parameter partials (23 used)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float v) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float rcp_a(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float lg2_a(float v) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float2 ex2x2(float2 v) { return make_float2(ex2(v.x), ex2(v.y)); }
__device__ __forceinline__ float2 f2b(float v) { return make_float2(v, v); }

// 1 / (1 + e^-v)
__device__ __forceinline__ float sigmoid_f(float v) { return rcp_a(1.0f + ex2(-v * LOG2E)); }

// log(1 + e^v) = max(v, 0) + log1p(e^-|v|); log1p(e) for e in (0, 1] from
// the series e - e^2/2 + e^3/3 below 2^-6 (truncation < e^3/4 relative),
// else log2(1 + e) ln 2.
__device__ __forceinline__ float softplus_f(float v) {
  const float e = ex2(-fabsf(v) * LOG2E);
  const float series = e * fmaf(e, fmaf(e, 0.33333334f, -0.5f), 1.0f);
  const float lg = lg2_a(1.0f + e) * LN2;
  return fmaxf(v, 0.0f) + (e < 0.015625f ? series : lg);
}

template <typename T> struct Act;
template <> struct Act<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
  static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
};
template <> struct Act<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  int n = valid ? 16 : 0;  // 0 bytes read: the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---- tensor memory (tcgen05): per-thread row storage ----
// A CTA of 4 warps owns tensor-memory lanes 0..127 (warp w: lanes 32w..32w+31,
// one lane per thread).  32x32b accesses move 16 consecutive 32-bit columns
// of the calling thread's lane.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float2 (&v)[NS / 2]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y),
      "f"(v[3].x), "f"(v[3].y), "f"(v[4].x), "f"(v[4].y), "f"(v[5].x), "f"(v[5].y), "f"(v[6].x),
      "f"(v[6].y), "f"(v[7].x), "f"(v[7].y) : "memory");
}
// Load and wait in one statement, so no use of the registers can be placed
// between the asynchronous load and its completion.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float2 (&v)[NS / 2]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y),
        "=f"(v[3].x), "=f"(v[3].y), "=f"(v[4].x), "=f"(v[4].y), "=f"(v[5].x), "=f"(v[5].y),
        "=f"(v[6].x), "=f"(v[6].y), "=f"(v[7].x), "=f"(v[7].y) : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float2 (&v)[4]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
      ::"r"(taddr), "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y),
      "f"(v[3].x), "f"(v[3].y) : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float2 (&v)[4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y),
        "=f"(v[3].x), "=f"(v[3].y) : "r"(taddr) : "memory");
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running; grid_dep_wait() returns once that kernel has completed and its
// memory is visible (immediately when there is no such dependency).
// grid_dep_trigger() lets the next such kernel start launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Stage rows [t_first, t_first + rows) x channels [d0, d0 + G) of a
// [B, T_, D] tensor of element type T into dst[rows][G]; rows outside
// [0, t_limit) and channels >= D read as zero.  NT threads cooperate.
template <typename T, int G, int NT>
__device__ __forceinline__ void stage_rows(T* dst, const T* src, int b, int t_first, int rows,
                                           int T_, int t_limit, int D, int d0, int tid) {
  constexpr int EPC = 16 / sizeof(T);
  constexpr int CPR = G / EPC;
  const int n = rows * CPR;
  for (int i = tid; i < n; i += NT) {
    const int r = i / CPR, cc = i - r * CPR;
    const int t = t_first + r, dd = d0 + cc * EPC;
    const bool ok = (t >= 0) && (t < t_limit) && (dd < D);
    const T* g = ok ? src + ((size_t)b * T_ + t) * D + dd : src;
    cp_async16(dst + r * G + cc * EPC, g, ok);
  }
}

// Stage rows [t_first, t_first + rows) of a [B, T_, NN] tensor whose rows
// are ld elements apart into dst[rows][NN]; rows outside [0, t_limit) read
// as zero.
template <typename T, int NT, int NN = NS>
__device__ __forceinline__ void stage_bc(T* dst, const T* src, int b, int t_first, int rows,
                                         int T_, int t_limit, int ld, int tid) {
  constexpr int EPC = 16 / sizeof(T);
  constexpr int CPR = NN / EPC;
  const int n = rows * CPR;
  for (int i = tid; i < n; i += NT) {
    const int r = i / CPR, cc = i - r * CPR;
    const int t = t_first + r;
    const bool ok = (t >= 0) && (t < t_limit);
    const T* g = ok ? src + ((size_t)b * T_ + t) * ld + cc * EPC : src;
    cp_async16(dst + r * NN + cc * EPC, g, ok);
  }
}

// ---------------------------------------------------------------------------
// geometry and kernel arguments
// ---------------------------------------------------------------------------

struct Geo {
  int B, T, D, K, nc, S, m;  // S segments of m chunks (the last may be short)
  int ldbc, lddbc;           // row strides (elements) of Bm/Cm and of dB/dC
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct FwdArgs {
  Geo g;
  const void *x, *dr, *z, *Bm, *Cm;
  const float *conv_w, *conv_b, *dt_bias, *a_log, *Dp;
  void *gated, *y_dbg;
  float* ckpt;
  float *agg_h, *agg_s;
  // carried state (all nullable): h before step 0 [B, 16, D] f32, the conv
  // inputs of steps -3..-1 [B, 3, D] act, and the same two after the window
  const float* h_in;
  const void* conv_in;
  float* h_out;
  void* conv_out;
};

struct BwdArgs {
  Geo g;
  const void *x, *dr, *z, *Bm, *Cm, *dg;
  const float *conv_w, *conv_b, *dt_bias, *a_log, *Dp, *ckpt;
  void *dx, *ddr, *dz, *du_dbg;
  float *dB, *dC;
  float *q, *sd, *dxpart, *dchead, *partials;
  float *d_conv_w, *d_conv_b, *d_dt_bias, *d_a_log, *dD;
  // carried state (all nullable): the forward's conv inputs of steps -3..-1
  // [B, 3, D] act; upstream gradients of the window's state outputs
  // (g_h [B, 16, D] f32, g_conv [B, 3, D] act); gradients of the state
  // inputs (d_h_in f32, d_conv_in act)
  const void* conv_in;
  const float* g_h;
  const void* g_conv;
  float* d_h_in;
  void* d_conv_in;
  int accumulate;
  uint32_t tcols;  // tensor-memory columns per CTA for the state history
};

// Forward shared memory: two staging buffers {x, delta_raw, z: [TT][GF]
// act; B, C: [TT][16] act}, B and C of the current tile as float [TT][16],
// and per-step scalars of one sub-tile sc[SUB][GF] float4 (thread-private
// slots: delta, delta*u, D*u, silu(z)).
struct FwdSmem {
  size_t x, dr, z, Bt, Ct, tile, fB, fC, sc, total;
};
__host__ __device__ inline FwdSmem fwd_smem(int es) {
  FwdSmem s;
  s.x = 0;
  s.dr = s.x + align_up((size_t)TT * GF * es, 128);
  s.z = s.dr + align_up((size_t)TT * GF * es, 128);
  s.Bt = s.z + align_up((size_t)TT * GF * es, 128);
  s.Ct = s.Bt + align_up((size_t)TT * NS * es, 128);
  s.tile = s.Ct + align_up((size_t)TT * NS * es, 128);
  s.fB = 2 * s.tile;
  s.fC = s.fB + (size_t)TT * NS * 4;
  s.sc = s.fC + (size_t)TT * NS * 4;
  s.total = s.sc + (size_t)SUB * GF * 16;
  return s;
}

// Split forward shared memory (CH = 128 / (N / 8) channels): two staging
// buffers {x: [TT+3][CH] (three halo rows), delta_raw, z: [TT][CH]; B, C:
// [TT][N]}, float B and C of the tile, and per-step scalars sc[SUB][CH]
// float4 shared by the threads of a channel.
struct Fwd2Smem {
  size_t x, dr, z, Bt, Ct, tile, fB, fC, sc, total;
};
__host__ __device__ inline Fwd2Smem fwd2_smem(int es, int N) {
  const int CH = 128 / (N / 8);  // channels per block
  Fwd2Smem s;
  s.x = 0;
  s.dr = s.x + align_up((size_t)(TT + 3) * CH * es, 128);
  s.z = s.dr + align_up((size_t)TT * CH * es, 128);
  s.Bt = s.z + align_up((size_t)TT * CH * es, 128);
  s.Ct = s.Bt + align_up((size_t)TT * N * es, 128);
  s.tile = s.Ct + align_up((size_t)TT * N * es, 128);
  s.fB = 2 * s.tile;
  s.fC = s.fB + (size_t)TT * N * 4;
  s.sc = s.fC + (size_t)TT * N * 4;
  s.total = s.sc + (size_t)SUB * CH * 16;
  return s;
}

// Backward shared memory: two staging buffers {x: [K+3][GB] (three halo rows
// before the chunk), delta_raw, z, d_gated: [K][GB] act; B, C: [K][16] act;
// the chunk's start state ck: [16][GB] f32}; B and C of the current chunk as
// float (the recomputed states live in tensor memory, see m3_bwd_kernel);
// per-step scalars, two thread-private float4 slots per step: s0[K][GB] =
// (delta, delta*u, dy, dz factor -> sum_n A dh exp(delta A) h_{t-1}) and
// s1[K][GB] = (D*u -> sum_n dh B, sigmoid(delta_raw + dt_bias), sigmoid(c),
// c); per-warp dB/dC sums red[K][NWB][32].
struct BwdSmem {
  size_t x, dr, z, dg, Bt, Ct, ck, tile, fB, fC, scal, red, total;
};
__host__ __device__ inline BwdSmem bwd_smem(int K, int es) {
  BwdSmem s;
  s.x = 0;
  s.dr = s.x + align_up((size_t)(K + 3) * GB * es, 128);
  s.z = s.dr + align_up((size_t)K * GB * es, 128);
  s.dg = s.z + align_up((size_t)K * GB * es, 128);
  s.Bt = s.dg + align_up((size_t)K * GB * es, 128);
  s.Ct = s.Bt + align_up((size_t)K * NS * es, 128);
  s.ck = s.Ct + align_up((size_t)K * NS * es, 128);
  s.tile = s.ck + (size_t)NS * GB * 4;
  s.fB = 2 * s.tile;
  s.fC = s.fB + (size_t)K * NS * 4;
  s.scal = s.fC + (size_t)K * NS * 4;
  s.red = s.scal + (size_t)2 * K * GB * 16;
  s.total = s.red + (size_t)K * NWB * 32 * 4;
  return s;
}

// Split backward (CH = 128 / (N / 8) channels per block): the same staging
// buffers for CH channels and N-wide B and C; per-step scalars s0/s1
// [K][CH] float4 shared by the threads of a channel; the conv-input gradient
// of the chunk's steps and of the next chunk's first three, dcs[K+3][CH];
// per-warp dB/dC sums red[K][4][2N].
struct Bwd2Smem {
  size_t x, dr, z, dg, Bt, Ct, ck, tile, fB, fC, scal, dcs, red, total;
};
__host__ __device__ inline Bwd2Smem bwd2_smem(int K, int es, int N) {
  const int CH = 128 / (N / 8);  // channels per block
  Bwd2Smem s;
  s.x = 0;
  s.dr = s.x + align_up((size_t)(K + 3) * CH * es, 128);
  s.z = s.dr + align_up((size_t)K * CH * es, 128);
  s.dg = s.z + align_up((size_t)K * CH * es, 128);
  s.Bt = s.dg + align_up((size_t)K * CH * es, 128);
  s.Ct = s.Bt + align_up((size_t)K * N * es, 128);
  s.ck = s.Ct + align_up((size_t)K * N * es, 128);
  s.tile = s.ck + (size_t)N * CH * 4;
  s.fB = 2 * s.tile;
  s.fC = s.fB + (size_t)K * N * 4;
  s.scal = s.fC + (size_t)K * N * 4;
  s.dcs = s.scal + (size_t)2 * K * CH * 16;
  s.red = s.dcs + align_up((size_t)(K + 3) * CH * 4, 128);
  s.total = s.red + (size_t)K * 4 * 2 * N * 4;
  return s;
}

// Backward aggregate shared memory: two buffers {delta_raw, z, d_gated:
// [TT][GB]; C: [TT][16]}, float C and per-step (delta, dy) [TT][GB] float2.
struct AggSmem {
  size_t dr, z, dg, Ct, tile, fC, sc, total;
};
__host__ __device__ inline AggSmem agg_smem(int es, int N = NS) {
  AggSmem s;
  s.dr = 0;
  s.z = s.dr + align_up((size_t)TT * GB * es, 128);
  s.dg = s.z + align_up((size_t)TT * GB * es, 128);
  s.Ct = s.dg + align_up((size_t)TT * GB * es, 128);
  s.tile = s.Ct + align_up((size_t)TT * N * es, 128);
  s.fC = 2 * s.tile;
  s.sc = s.fC + (size_t)TT * N * 4;
  s.total = s.sc + (size_t)TT * GB * 8;
  return s;
}

// ---------------------------------------------------------------------------
// forward: FINAL = run each segment from its true start state, write gated
// (+y) and a checkpoint every K steps; !FINAL = local pass from zero over
// segments 0..S-2 writing only the end state and the summed step size.
// Lanes are handled in pairs with packed f32x2 arithmetic.
// ---------------------------------------------------------------------------

template <typename T, bool FINAL>
__global__ void __launch_bounds__(GF) m3_fwd_kernel(FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Geo g = a.g;
  const int tid = threadIdx.x;
  const int d0 = blockIdx.x * GF;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int d = d0 + tid;
  const bool active = d < g.D;
  const int c_begin = s * g.m;
  const int c_end = min(c_begin + g.m, g.nc);
  const int t_begin = c_begin * g.K;
  const int t_end = min(c_end * g.K, g.T);
  const FwdSmem L = fwd_smem(sizeof(T));
  const T* xg = static_cast<const T*>(a.x);
  const T* drg = static_cast<const T*>(a.dr);
  const T* zg = static_cast<const T*>(a.z);
  const T* Bg = static_cast<const T*>(a.Bm);
  const T* Cg = static_cast<const T*>(a.Cm);
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);

  auto stage = [&](int t0, int buf) {
    unsigned char* base = smem + (size_t)buf * L.tile;
    stage_rows<T, GF, GF>(reinterpret_cast<T*>(base + L.x), xg, b, t0, TT, g.T, t_end, g.D, d0, tid);
    stage_rows<T, GF, GF>(reinterpret_cast<T*>(base + L.dr), drg, b, t0, TT, g.T, t_end, g.D, d0, tid);
    stage_bc<T, GF>(reinterpret_cast<T*>(base + L.Bt), Bg, b, t0, TT, g.T, t_end, g.ldbc, tid);
    if (FINAL) {
      stage_rows<T, GF, GF>(reinterpret_cast<T*>(base + L.z), zg, b, t0, TT, g.T, t_end, g.D, d0, tid);
      stage_bc<T, GF>(reinterpret_cast<T*>(base + L.Ct), Cg, b, t0, TT, g.T, t_end, g.ldbc, tid);
    }
    cp_async_commit();
  };
  stage(t_begin, 0);  // first tile in flight while the parameters and carries load
  if (!FINAL) grid_dep_trigger();

  float2 a2[NS / 2];  // A log2(e) for lanes (2i, 2i+1)
#pragma unroll
  for (int i = 0; i < NS / 2; ++i) {
    a2[i].x = active ? -expf(a.a_log[(size_t)d * NS + 2 * i]) * LOG2E : 0.f;
    a2[i].y = active ? -expf(a.a_log[(size_t)d * NS + 2 * i + 1]) * LOG2E : 0.f;
  }
  float w[WC];
#pragma unroll
  for (int k = 0; k < WC; ++k) w[k] = active ? a.conv_w[(size_t)d * WC + k] : 0.f;
  const float cb = active ? a.conv_b[d] : 0.f;
  const float dtb = active ? a.dt_bias[d] : 0.f;
  const float Dd = active ? a.Dp[d] : 0.f;

  float2 h[NS / 2];
#pragma unroll
  for (int i = 0; i < NS / 2; ++i) h[i] = make_float2(0.f, 0.f);
  if (FINAL && a.h_in && active) {  // the local passes start from zero
    const float* h0 = a.h_in + (size_t)b * NS * g.D + d;
#pragma unroll
    for (int i = 0; i < NS / 2; ++i) h[i] = make_float2(h0[(size_t)(2 * i) * g.D], h0[(size_t)(2 * i + 1) * g.D]);
  }
  if (FINAL && s > 0) {
    grid_dep_wait();  // the aggregate pass's outputs
    // The scan is linear in the state: chain the earlier segments' local end
    // states with their decays, start(s'+1) = exp(A sum delta_s') start(s') +
    // local_end(s'), to get this segment's true start state.
    const float* __restrict__ agg_s = a.agg_s;
    const float* __restrict__ agg_h = a.agg_h;
#pragma unroll 4
    for (int sp = 0; sp < s; ++sp) {
      const size_t bs = (size_t)b * g.S + sp;
      const float2 dl2 = f2b(active ? agg_s[bs * g.D + d] : 0.f);
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        const float* ah = agg_h + (bs * NS + 2 * i) * g.D + d;
        const float2 loc = active ? make_float2(ah[0], ah[g.D]) : make_float2(0.f, 0.f);
        h[i] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[i])), h[i], loc);
      }
    }
  }

  // conv window x[t-3], x[t-2], x[t-1]; steps before 0 come from the
  // carried conv inputs (row step + 3), zero without them
  auto x_at = [&](int t) -> float {
    if (t >= 0) return Act<T>::ld(xg + ((size_t)b * g.T + t) * g.D + d);
    if (a.conv_in) return Act<T>::ld(static_cast<const T*>(a.conv_in) + ((size_t)b * 3 + t + 3) * g.D + d);
    return 0.f;
  };
  float xm3 = 0.f, xm2 = 0.f, xm1 = 0.f;
  if (active) {
    xm3 = x_at(t_begin - 3);
    xm2 = x_at(t_begin - 2);
    xm1 = x_at(t_begin - 1);
  }
  float sdelta = 0.f;


  float4* scs = reinterpret_cast<float4*>(smem + L.sc) + tid;  // this thread's slots, stride GF
  int kc = 0;  // steps left until the next checkpoint
  for (int t0 = t_begin, it = 0; t0 < t_end; t0 += TT, ++it) {
    const int buf = it & 1;
    if (t0 + TT < t_end) {
      stage(t0 + TT, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const unsigned char* base = smem + (size_t)buf * L.tile;
    {
      const T* Bt = reinterpret_cast<const T*>(base + L.Bt);
      const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
      for (int i = tid; i < TT * NS; i += GF) {
        fB[i] = Act<T>::ld(Bt + i);
        if (FINAL) fC[i] = Act<T>::ld(Ct + i);
      }
    }
    __syncthreads();
    const T* xt = reinterpret_cast<const T*>(base + L.x);
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const int steps = min(TT, t_end - t0);
    for (int j0 = 0; j0 < steps; j0 += SUB) {
      const int ns = min(SUB, steps - j0);
      // scalar pass: independent per step (conv, SiLU, softplus, gate factor)
#pragma unroll 4
      for (int j = 0; j < ns; ++j) {
        const float xv = Act<T>::ld(xt + (j0 + j) * GF + tid);
        const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
        xm3 = xm2;
        xm2 = xm1;
        xm1 = xv;
        const float u = cpre * sigmoid_f(cpre);
        const float delta = softplus_f(Act<T>::ld(drt + (j0 + j) * GF + tid) + dtb);
        float gz = 0.f;
        if (FINAL) {
          const float zv = Act<T>::ld(zt + (j0 + j) * GF + tid);
          gz = zv * sigmoid_f(zv);
        } else {
          sdelta += delta;
        }
        scs[j * GF] = make_float4(delta, delta * u, Dd * u, gz);
      }
      // state pass: the only loop-carried dependence is h
#pragma unroll 4
      for (int j = 0; j < ns; ++j) {
        if (FINAL) {
          if (kc == 0) {
            const int t = t0 + j0 + j;
            if (active) {
              float* ck = a.ckpt + (((size_t)b * g.nc + t / g.K) * NS) * g.D + d;
#pragma unroll
              for (int i = 0; i < NS / 2; ++i) {
                ck[(size_t)(2 * i) * g.D] = h[i].x;
                ck[(size_t)(2 * i + 1) * g.D] = h[i].y;
              }
            }
            kc = g.K;
          }
          --kc;
        }
        const float4 v = scs[j * GF];
        const float2 dl2 = f2b(v.x);
        const float2 du2 = f2b(v.y);
        const float4* B4 = reinterpret_cast<const float4*>(fB + (j0 + j) * NS);
        if (FINAL) {
          const float4* C4 = reinterpret_cast<const float4*>(fC + (j0 + j) * NS);
          float2 y01 = make_float2(0.f, 0.f), y23 = make_float2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 bv = B4[q];
            const float4 cv = C4[q];
            const float2 dA0 = ex2x2(__fmul2_rn(dl2, a2[2 * q]));
            const float2 dA1 = ex2x2(__fmul2_rn(dl2, a2[2 * q + 1]));
            h[2 * q] = __ffma2_rn(dA0, h[2 * q], __fmul2_rn(du2, make_float2(bv.x, bv.y)));
            h[2 * q + 1] = __ffma2_rn(dA1, h[2 * q + 1], __fmul2_rn(du2, make_float2(bv.z, bv.w)));
            y01 = __ffma2_rn(make_float2(cv.x, cv.y), h[2 * q], y01);
            y23 = __ffma2_rn(make_float2(cv.z, cv.w), h[2 * q + 1], y23);
          }
          const float y = ((y01.x + y01.y) + (y23.x + y23.y)) + v.z;
          if (active) {
            const size_t i = ((size_t)b * g.T + t0 + j0 + j) * g.D + d;
            Act<T>::st(static_cast<T*>(a.gated) + i, y * v.w);
            if (a.y_dbg) Act<T>::st(static_cast<T*>(a.y_dbg) + i, y);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 bv = B4[q];
            const float2 dA0 = ex2x2(__fmul2_rn(dl2, a2[2 * q]));
            const float2 dA1 = ex2x2(__fmul2_rn(dl2, a2[2 * q + 1]));
            h[2 * q] = __ffma2_rn(dA0, h[2 * q], __fmul2_rn(du2, make_float2(bv.x, bv.y)));
            h[2 * q + 1] = __ffma2_rn(dA1, h[2 * q + 1], __fmul2_rn(du2, make_float2(bv.z, bv.w)));
          }
        }
      }
    }
    __syncthreads();
  }
  if (FINAL && s == g.S - 1 && active) {
    if (a.h_out) {
      float* ho = a.h_out + (size_t)b * NS * g.D + d;
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        ho[(size_t)(2 * i) * g.D] = h[i].x;
        ho[(size_t)(2 * i + 1) * g.D] = h[i].y;
      }
    }
    if (a.conv_out) {  // the window now holds x[T-3], x[T-2], x[T-1]
      T* co = static_cast<T*>(a.conv_out) + (size_t)b * 3 * g.D + d;
      Act<T>::st(co, xm3);
      Act<T>::st(co + g.D, xm2);
      Act<T>::st(co + 2 * (size_t)g.D, xm1);
    }
  }
  if (!FINAL && active) {
    float* ah = a.agg_h + (((size_t)b * g.S + s) * NS) * g.D + d;
#pragma unroll
    for (int i = 0; i < NS / 2; ++i) {
      ah[(size_t)(2 * i) * g.D] = h[i].x;
      ah[(size_t)(2 * i + 1) * g.D] = h[i].y;
    }
    a.agg_s[((size_t)b * g.S + s) * g.D + d] = sdelta;
  }
}

// ---------------------------------------------------------------------------
// forward with the lanes split over N / 8 threads per channel (8 lanes
// each; 128 / (N / 8) channels per block): the threads of a channel take the
// scalar pass of every (N / 8)-th step and sum y with shuffles.  For d_state
// 32 and 64, and for d_state-16 grids that fill less than one wave; the same
// results as m3_fwd_kernel up to the order of f32 sums.
// ---------------------------------------------------------------------------

template <typename T, bool FINAL, int N>
__global__ void __launch_bounds__(128) m3_fwd2_kernel(FwdArgs a) {
  constexpr int G = N / 8;     // threads per channel
  constexpr int CH = 128 / G;  // channels per block
  extern __shared__ __align__(128) unsigned char smem[];
  const Geo g = a.g;
  const int tid = threadIdx.x;
  const int hf = tid % G;   // this thread's state lanes: 8 hf .. 8 hf + 7
  const int ch = tid / G;   // channel within the block
  const int d0 = blockIdx.x * CH;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int d = d0 + ch;
  const bool active = d < g.D;
  const int c_begin = s * g.m;
  const int c_end = min(c_begin + g.m, g.nc);
  const int t_begin = c_begin * g.K;
  const int t_end = min(c_end * g.K, g.T);
  const Fwd2Smem L = fwd2_smem(sizeof(T), N);
  const T* xg = static_cast<const T*>(a.x);
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);

  // x is staged with the three steps before the tile (row r = step t0 - 3 + r)
  auto stage = [&](int t0, int buf) {
    unsigned char* base = smem + (size_t)buf * L.tile;
    stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.x), xg, b, t0 - 3, TT + 3, g.T, t_end, g.D, d0, tid);
    stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.dr), static_cast<const T*>(a.dr), b, t0, TT, g.T, t_end, g.D, d0, tid);
    stage_bc<T, 128, N>(reinterpret_cast<T*>(base + L.Bt), static_cast<const T*>(a.Bm), b, t0, TT, g.T, t_end, g.ldbc, tid);
    if (FINAL) {
      stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.z), static_cast<const T*>(a.z), b, t0, TT, g.T, t_end, g.D, d0, tid);
      stage_bc<T, 128, N>(reinterpret_cast<T*>(base + L.Ct), static_cast<const T*>(a.Cm), b, t0, TT, g.T, t_end, g.ldbc, tid);
    }
    cp_async_commit();
  };
  stage(t_begin, 0);
  if (!FINAL) grid_dep_trigger();

  float2 a2[4];  // A log2(e) of lanes (8 hf + 2 P, 8 hf + 2 P + 1)
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    const int n = 8 * hf + 2 * P;
    a2[P].x = active ? -expf(a.a_log[(size_t)d * N + n]) * LOG2E : 0.f;
    a2[P].y = active ? -expf(a.a_log[(size_t)d * N + n + 1]) * LOG2E : 0.f;
  }
  float w[WC];
#pragma unroll
  for (int k = 0; k < WC; ++k) w[k] = active ? a.conv_w[(size_t)d * WC + k] : 0.f;
  const float cb = active ? a.conv_b[d] : 0.f;
  const float dtb = active ? a.dt_bias[d] : 0.f;
  const float Dd = active ? a.Dp[d] : 0.f;

  float2 h[4];
#pragma unroll
  for (int P = 0; P < 4; ++P) h[P] = make_float2(0.f, 0.f);
  if (FINAL && a.h_in && active) {
    const float* h0 = a.h_in + (size_t)b * N * g.D + d;
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      const int n = 8 * hf + 2 * P;
      h[P] = make_float2(h0[(size_t)n * g.D], h0[(size_t)(n + 1) * g.D]);
    }
  }
  if (FINAL && s > 0) {
    grid_dep_wait();  // the aggregate pass's outputs
#pragma unroll 2
    for (int sp = 0; sp < s; ++sp) {
      const size_t bs = (size_t)b * g.S + sp;
      const float2 dl2 = f2b(active ? a.agg_s[bs * g.D + d] : 0.f);
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const float* ah = a.agg_h + (bs * N + 8 * hf + 2 * P) * g.D + d;
        const float2 loc = active ? make_float2(ah[0], ah[g.D]) : make_float2(0.f, 0.f);
        h[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), h[P], loc);
      }
    }
  }
  float sdelta = 0.f;
  float4* scs = reinterpret_cast<float4*>(smem + L.sc) + ch;  // shared by the channel's threads, stride CH
  int kc = 0;  // steps left until the next checkpoint
  for (int t0 = t_begin, it = 0; t0 < t_end; t0 += TT, ++it) {
    const int buf = it & 1;
    if (t0 + TT < t_end) {
      stage(t0 + TT, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    unsigned char* base = smem + (size_t)buf * L.tile;
    if (a.conv_in && t0 < 3 && active && hf == 0) {
      // halo rows before step 0 (staged as zeros): the carried conv inputs
      T* xw = reinterpret_cast<T*>(base + L.x);
      const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * g.D + d;
      for (int r = 0; r < 3 - t0; ++r) xw[r * CH + ch] = ci[(size_t)(t0 + r) * g.D];
    }
    {
      const T* Bt = reinterpret_cast<const T*>(base + L.Bt);
      const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
      for (int i = tid; i < TT * N; i += 128) {
        fB[i] = Act<T>::ld(Bt + i);
        if (FINAL) fC[i] = Act<T>::ld(Ct + i);
      }
    }
    __syncthreads();
    const T* xt = reinterpret_cast<const T*>(base + L.x);
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const int steps = min(TT, t_end - t0);
    for (int j0 = 0; j0 < steps; j0 += SUB) {
      const int ns = min(SUB, steps - j0);
      // scalar pass, this thread's steps (every G-th)
#pragma unroll 2
      for (int j = hf; j < ns; j += G) {
        const int r = j0 + j;
        const float xm3 = Act<T>::ld(xt + r * CH + ch);
        const float xm2 = Act<T>::ld(xt + (r + 1) * CH + ch);
        const float xm1 = Act<T>::ld(xt + (r + 2) * CH + ch);
        const float xv = Act<T>::ld(xt + (r + 3) * CH + ch);
        const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
        const float u = cpre * sigmoid_f(cpre);
        const float delta = softplus_f(Act<T>::ld(drt + r * CH + ch) + dtb);
        float gz = 0.f;
        if (FINAL) {
          const float zv = Act<T>::ld(zt + r * CH + ch);
          gz = zv * sigmoid_f(zv);
        }
        scs[j * CH] = make_float4(delta, delta * u, Dd * u, gz);
      }
      __syncwarp();
      // state pass, both threads
#pragma unroll 4
      for (int j = 0; j < ns; ++j) {
        if (FINAL) {
          if (kc == 0) {
            const int t = t0 + j0 + j;
            if (active) {
              float* ck = a.ckpt + (((size_t)b * g.nc + t / g.K) * N + 8 * hf) * g.D + d;
#pragma unroll
              for (int P = 0; P < 4; ++P) {
                ck[(size_t)(2 * P) * g.D] = h[P].x;
                ck[(size_t)(2 * P + 1) * g.D] = h[P].y;
              }
            }
            kc = g.K;
          }
          --kc;
        }
        const float4 v = scs[j * CH];
        const float2 dl2 = f2b(v.x);
        const float2 du2 = f2b(v.y);
        const float* Bj = fB + (j0 + j) * N + 8 * hf;
        if (FINAL) {
          const float* Cj = fC + (j0 + j) * N + 8 * hf;
          float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int P = 0; P < 4; ++P) {
            const float2 bb = *reinterpret_cast<const float2*>(Bj + 2 * P);
            const float2 cc = *reinterpret_cast<const float2*>(Cj + 2 * P);
            h[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), h[P], __fmul2_rn(du2, bb));
            y2 = __ffma2_rn(cc, h[P], y2);
          }
          float y = y2.x + y2.y;
#pragma unroll
          for (int o = 1; o < G; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
          y += v.z;
          if (active && hf == j % G) {
            const size_t i = ((size_t)b * g.T + t0 + j0 + j) * g.D + d;
            Act<T>::st(static_cast<T*>(a.gated) + i, y * v.w);
            if (a.y_dbg) Act<T>::st(static_cast<T*>(a.y_dbg) + i, y);
          }
        } else {
          sdelta += v.x;
#pragma unroll
          for (int P = 0; P < 4; ++P) {
            const float2 bb = *reinterpret_cast<const float2*>(Bj + 2 * P);
            h[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), h[P], __fmul2_rn(du2, bb));
          }
        }
      }
      __syncwarp();  // this sub-tile's slots are read; the next one overwrites them
    }
    __syncthreads();
  }
  if (FINAL && s == g.S - 1 && active) {
    if (a.h_out) {
      float* ho = a.h_out + ((size_t)b * N + 8 * hf) * g.D + d;
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        ho[(size_t)(2 * P) * g.D] = h[P].x;
        ho[(size_t)(2 * P + 1) * g.D] = h[P].y;
      }
    }
    if (a.conv_out && hf == 0) {  // the conv inputs of steps T-3 .. T-1
      T* co = static_cast<T*>(a.conv_out) + (size_t)b * 3 * g.D + d;
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int t = g.T - 3 + r;
        float v = 0.f;
        if (t >= 0)
          v = Act<T>::ld(xg + ((size_t)b * g.T + t) * g.D + d);
        else if (a.conv_in)
          v = Act<T>::ld(static_cast<const T*>(a.conv_in) + ((size_t)b * 3 + t + 3) * g.D + d);
        Act<T>::st(co + (size_t)r * g.D, v);
      }
    }
  }
  if (!FINAL && active) {
    float* ah = a.agg_h + (((size_t)b * g.S + s) * N + 8 * hf) * g.D + d;
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      ah[(size_t)(2 * P) * g.D] = h[P].x;
      ah[(size_t)(2 * P + 1) * g.D] = h[P].y;
    }
    if (hf == 0) a.agg_s[((size_t)b * g.S + s) * g.D + d] = sdelta;
  }
}

// ---------------------------------------------------------------------------
// backward aggregate (segments 1..S-1): the adjoint carry a segment passes to
// its predecessor when nothing enters it from the right,
//   carry_t = exp(delta_t A) * (dy_t C_t + carry_{t+1}),
// and the summed step size (the segment's total decay).
// ---------------------------------------------------------------------------

// TPC threads per channel: one (16 lanes each, d_state 16) or d_state / 8
// (8 lanes each, 128 / TPC channels per block), the threads of a channel
// taking the scalar pass of every TPC-th step.
template <typename T, int TPC, int N>
__global__ void __launch_bounds__(GB) m3_bwd_agg_kernel(BwdArgs a) {
  constexpr int G = GB / TPC;        // channels per block
  constexpr int NL = N / TPC;        // state lanes per thread
  extern __shared__ __align__(128) unsigned char smem[];
  const Geo g = a.g;
  const int tid = threadIdx.x;
  const int hf = tid % TPC;
  const int ch = tid / TPC;
  const int d0 = blockIdx.x * G;
  const int s = blockIdx.y + 1;
  const int b = blockIdx.z;
  const int d = d0 + ch;
  const bool active = d < g.D;
  const int t_begin = s * g.m * g.K;
  const int t_end = min((s + 1) * g.m * g.K, g.T);
  const AggSmem L = agg_smem(sizeof(T), N);
  float* fC = reinterpret_cast<float*>(smem + L.fC);
  const int ntiles = (t_end - t_begin + TT - 1) / TT;
  auto tile_start = [&](int i) { return max(t_begin, t_end - (i + 1) * TT); };
  auto stage = [&](int i, int buf) {
    unsigned char* base = smem + (size_t)buf * L.tile;
    const int t0 = tile_start(i);
    const int rows = (t_end - i * TT) - t0;
    stage_rows<T, G, GB>(reinterpret_cast<T*>(base + L.dr), static_cast<const T*>(a.dr), b, t0, rows, g.T, g.T, g.D, d0, tid);
    stage_rows<T, G, GB>(reinterpret_cast<T*>(base + L.z), static_cast<const T*>(a.z), b, t0, rows, g.T, g.T, g.D, d0, tid);
    stage_rows<T, G, GB>(reinterpret_cast<T*>(base + L.dg), static_cast<const T*>(a.dg), b, t0, rows, g.T, g.T, g.D, d0, tid);
    stage_bc<T, GB, N>(reinterpret_cast<T*>(base + L.Ct), static_cast<const T*>(a.Cm), b, t0, rows, g.T, g.T, g.ldbc, tid);
    cp_async_commit();
  };

  stage(0, 0);  // first tile in flight while the parameters load
  grid_dep_trigger();

  float2 a2[NL / 2];
#pragma unroll
  for (int i = 0; i < NL / 2; ++i) {
    const int n = NL * hf + 2 * i;
    a2[i].x = active ? -expf(a.a_log[(size_t)d * N + n]) * LOG2E : 0.f;
    a2[i].y = active ? -expf(a.a_log[(size_t)d * N + n + 1]) * LOG2E : 0.f;
  }
  const float dtb = active ? a.dt_bias[d] : 0.f;
  float2 carry[NL / 2];
#pragma unroll
  for (int i = 0; i < NL / 2; ++i) carry[i] = make_float2(0.f, 0.f);
  float sdelta = 0.f;

  {
    // dB and dC are sums over channel groups (global reductions in the main
    // kernel): this kernel runs before it, so it clears them.
    const size_t ncta = (size_t)gridDim.x * gridDim.y * gridDim.z;
    const size_t cid = blockIdx.x + (size_t)gridDim.x * (blockIdx.y + (size_t)gridDim.y * blockIdx.z);
    const size_t total = (size_t)g.B * g.T * N;
    for (size_t i = cid * GB + tid; i < total; i += ncta * GB) {
      const size_t o = (i / N) * g.lddbc + (i % N);
      a.dB[o] = 0.f;
      a.dC[o] = 0.f;
    }
  }
  for (int i = 0; i < ntiles; ++i) {
    const int buf = i & 1;
    if (i + 1 < ntiles) {
      stage(i + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const unsigned char* base = smem + (size_t)buf * L.tile;
    const int t0 = tile_start(i);
    const int steps = (t_end - i * TT) - t0;
    {
      const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
      for (int k = tid; k < steps * N; k += GB) fC[k] = Act<T>::ld(Ct + k);
    }
    __syncthreads();
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const T* dgt = reinterpret_cast<const T*>(base + L.dg);
    float2* scs = reinterpret_cast<float2*>(smem + L.sc) + ch;  // per channel, stride G
#pragma unroll 4
    for (int j = hf; j < steps; j += TPC) {  // scalar pass
      const float zv = Act<T>::ld(zt + j * G + ch);
      const float dy = Act<T>::ld(dgt + j * G + ch) * zv * sigmoid_f(zv);
      const float delta = softplus_f(Act<T>::ld(drt + j * G + ch) + dtb);
      scs[j * G] = make_float2(delta, dy);
    }
    if (TPC > 1) __syncwarp();
#pragma unroll 4
    for (int j = steps - 1; j >= 0; --j) {  // state pass
      const float2 v = scs[j * G];
      sdelta += v.x;
      const float2 dl2 = f2b(v.x);
      const float2 dy2 = f2b(v.y);
      const float2* C2 = reinterpret_cast<const float2*>(fC + j * N + NL * hf);
#pragma unroll
      for (int q = 0; q < NL / 2; ++q) {
        carry[q] = __fmul2_rn(ex2x2(__fmul2_rn(dl2, a2[q])), __ffma2_rn(dy2, C2[q], carry[q]));
      }
    }
    __syncthreads();
  }
  if (active) {
    const size_t bs = (size_t)b * g.S + s;
#pragma unroll
    for (int i = 0; i < NL / 2; ++i) {
      a.q[(bs * N + NL * hf + 2 * i) * g.D + d] = carry[i].x;
      a.q[(bs * N + NL * hf + 2 * i + 1) * g.D + d] = carry[i].y;
    }
    if (hf == 0) a.sd[bs * g.D + d] = sdelta;
  }
}

// ---------------------------------------------------------------------------
// backward main kernel
//
// Each thread keeps its 16 state lanes in 4 quads whose order is rotated by
// the lane's two low bits: register quad qs holds state quad qs ^ (lane & 3).
// The dB/dC sum over the warp's 32 channels then starts with two
// butterfly levels that need no selects (partners hold the same state lane
// in the same register), as the reduce-scatter below relies on.
// ---------------------------------------------------------------------------

// Sum over the 32 lanes of v[0..15] (v[s] holds state lane
// 4 * ((s >> 2) ^ (lane & 3)) + (s & 3)); returns the total for state lane
// 4 * (lane & 3) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1).
__device__ __forceinline__ float warp_sum16_rotated(float (&v)[NS], int lane) {
#pragma unroll
  for (int s = 0; s < 8; ++s) v[s] += __shfl_xor_sync(0xffffffffu, v[s + 8], 2);
#pragma unroll
  for (int s = 0; s < 4; ++s) v[s] += __shfl_xor_sync(0xffffffffu, v[s + 4], 1);
  {
    const bool up = (lane & 8) != 0;
    const float s0 = up ? v[0] : v[2], s1 = up ? v[1] : v[3];
    const float k0 = up ? v[2] : v[0], k1 = up ? v[3] : v[1];
    v[0] = k0 + __shfl_xor_sync(0xffffffffu, s0, 8);
    v[1] = k1 + __shfl_xor_sync(0xffffffffu, s1, 8);
  }
  {
    const bool up = (lane & 4) != 0;
    const float s0 = up ? v[0] : v[1];
    const float k0 = up ? v[1] : v[0];
    v[0] = k0 + __shfl_xor_sync(0xffffffffu, s0, 4);
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// ST: compiled with the carried-state terms; the plain entry points run the
// instance without them.  SCAN: stop at du (written out) -- the SiLU and
// conv backward then run in m3_conv_bwd_kernel with du plus any gradient
// reaching u from outside the layer core.
template <typename T, bool ST, bool SCAN>
__global__ void __launch_bounds__(GB, 3) m3_bwd_kernel(BwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Geo g = a.g;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int rot = lane & 3;
  const int d0 = blockIdx.x * GB;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int d = d0 + tid;
  const bool active = d < g.D;
  const int c_begin = s * g.m;
  const int c_end = min(c_begin + g.m, g.nc);
  const int t_begin = c_begin * g.K;
  const int t_end = min(c_end * g.K, g.T);
  const int K = g.K;
  const BwdSmem L = bwd_smem(K, sizeof(T));
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);
  float* red = reinterpret_cast<float*>(smem + L.red);
  // state lane of register slot 2*i (pair i): quad (i >> 1) ^ rot, offset 2*(i & 1)
  auto lane_of = [&](int i) { return 4 * ((i >> 1) ^ rot) + 2 * (i & 1); };

  // The recomputed states of a chunk (K rows of 16 f32 per channel) live in
  // tensor memory: row j of this thread = columns [16 j, 16 j + 16) of its
  // lane.  Warp 0 allocates for the CTA; every exit path below deallocates.
  __shared__ uint32_t tmem_slot;
  if (warp == 0) tmem_alloc(&tmem_slot, a.tcols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t trow = tmem_slot + ((uint32_t)(warp * 32) << 16);

  float2 a2[NS / 2];
  float w[WC];
  float cb = 0.f, dtb = 0.f, Dd = 0.f;
#pragma unroll
  for (int i = 0; i < NS / 2; ++i) {
    const int n = lane_of(i);
    a2[i].x = active ? -expf(a.a_log[(size_t)d * NS + n]) * LOG2E : 0.f;
    a2[i].y = active ? -expf(a.a_log[(size_t)d * NS + n + 1]) * LOG2E : 0.f;
  }
#pragma unroll
  for (int k = 0; k < WC; ++k) w[k] = active ? a.conv_w[(size_t)d * WC + k] : 0.f;
  if (active) {
    cb = a.conv_b[d];
    dtb = a.dt_bias[d];
    Dd = a.Dp[d];
  }

  // adjoint carry entering the segment's last step from the right:
  // exp(delta_{t+1} A) dh_{t+1}
  float2 carry[NS / 2];
#pragma unroll
  for (int i = 0; i < NS / 2; ++i) carry[i] = make_float2(0.f, 0.f);
  if (ST && a.g_h && active) {  // the gradient of the state output enters after the last step
    const float* gh = a.g_h + (size_t)b * NS * g.D + d;
#pragma unroll
    for (int i = 0; i < NS / 2; ++i) {
      const int n = lane_of(i);
      carry[i] = make_float2(gh[(size_t)n * g.D], gh[(size_t)(n + 1) * g.D]);
    }
  }
  const T* xg = static_cast<const T*>(a.x);
  auto stage = [&](int c, int buf) {
    unsigned char* base = smem + (size_t)buf * L.tile;
    const int t0 = c * K;
    stage_rows<T, GB, GB>(reinterpret_cast<T*>(base + L.x), xg, b, t0 - 3, K + 3, g.T, g.T, g.D, d0, tid);
    stage_rows<T, GB, GB>(reinterpret_cast<T*>(base + L.dr), static_cast<const T*>(a.dr), b, t0, K, g.T, g.T, g.D, d0, tid);
    stage_rows<T, GB, GB>(reinterpret_cast<T*>(base + L.z), static_cast<const T*>(a.z), b, t0, K, g.T, g.T, g.D, d0, tid);
    stage_rows<T, GB, GB>(reinterpret_cast<T*>(base + L.dg), static_cast<const T*>(a.dg), b, t0, K, g.T, g.T, g.D, d0, tid);
    stage_bc<T, GB>(reinterpret_cast<T*>(base + L.Bt), static_cast<const T*>(a.Bm), b, t0, K, g.T, g.T, g.ldbc, tid);
    stage_bc<T, GB>(reinterpret_cast<T*>(base + L.Ct), static_cast<const T*>(a.Cm), b, t0, K, g.T, g.T, g.ldbc, tid);
    // chunk start state: 16 rows of GB floats from ckpt[b, c, :, d0:d0+GB]
    stage_rows<float, GB, GB>(reinterpret_cast<float*>(base + L.ck), a.ckpt + ((size_t)b * g.nc + c) * NS * g.D,
                              0, 0, NS, NS, NS, g.D, d0, tid);
    cp_async_commit();
  };

  stage(c_end - 1, 0);  // last chunk in flight while the carries load
  grid_dep_trigger();
  // the aggregate kernel's carries, and its clearing of dB and dC before
  // this kernel's reductions into them
  grid_dep_wait();
  if (s + 1 < g.S) {
    // chain the later segments right to left: in(s'-1) = exp(A sum delta_s')
    // in(s') + local(s'), with in(S-1) = 0
    const float* __restrict__ sd = a.sd;
    const float* __restrict__ q = a.q;
#pragma unroll 2
    for (int sp = g.S - 1; sp > s; --sp) {
      const size_t bs = (size_t)b * g.S + sp;
      const float2 dl2 = f2b(active ? sd[bs * g.D + d] : 0.f);
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        const float* qq = q + (bs * NS + lane_of(i)) * g.D + d;
        const float2 loc = active ? make_float2(qq[0], qq[g.D]) : make_float2(0.f, 0.f);
        carry[i] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[i])), carry[i], loc);
      }
    }
  }
  float2 dAp[NS / 2];  // dL/dA per lane
#pragma unroll
  for (int i = 0; i < NS / 2; ++i) dAp[i] = make_float2(0.f, 0.f);
  float dD_acc = 0.f, ddtb_acc = 0.f, dcb_acc = 0.f;
  float dcw[WC] = {0.f, 0.f, 0.f, 0.f};
  float dc1 = 0.f, dc2 = 0.f, dc3 = 0.f;  // conv-input gradient at t+1, t+2, t+3

  for (int c = c_end - 1; c >= c_begin; --c) {
    const int buf = (c_end - 1 - c) & 1;
    if (c - 1 >= c_begin) {
      stage(c - 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const unsigned char* base = smem + (size_t)buf * L.tile;
    if (ST && a.conv_in && c * K < 3 && active) {
      // halo rows before step 0 (staged as zeros): the carried conv inputs.
      // Only this thread reads its column of the x tile.
      T* xw = reinterpret_cast<T*>(smem + (size_t)buf * L.tile + L.x);
      const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * g.D + d;
      for (int r = 0; r < 3 - c * K; ++r) xw[r * GB + tid] = ci[(size_t)(c * K + r) * g.D];
    }
    {
      const T* Bt = reinterpret_cast<const T*>(base + L.Bt);
      const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
      for (int i = tid; i < K * NS; i += GB) {
        fB[i] = Act<T>::ld(Bt + i);
        fC[i] = Act<T>::ld(Ct + i);
      }
    }
    __syncthreads();
    const T* xt = reinterpret_cast<const T*>(base + L.x);  // row r is step c*K - 3 + r
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const T* dgt = reinterpret_cast<const T*>(base + L.dg);
    const float* ckt = reinterpret_cast<const float*>(base + L.ck);
    const int steps = min(K, g.T - c * K);

    float4* s0 = reinterpret_cast<float4*>(smem + L.scal) + tid;  // thread-private, stride GB
    float4* s1 = s0 + (size_t)K * GB;
    T* const dz_c = static_cast<T*>(a.dz) + ((size_t)b * g.T + (size_t)c * K) * g.D + d;
    T* const ddr_c = static_cast<T*>(a.ddr) + ((size_t)b * g.T + (size_t)c * K) * g.D + d;
    T* const dx_c = static_cast<T*>(a.dx) + ((size_t)b * g.T + (size_t)c * K) * g.D + d;
    T* const du_c = a.du_dbg ? static_cast<T*>(a.du_dbg) + ((size_t)b * g.T + (size_t)c * K) * g.D + d
                             : nullptr;

    // The four passes over the chunk.
    {
      const int nst = steps;

      // ---- scalar pass: everything per step that does not need the state ----
      {
        float xm3 = Act<T>::ld(xt + 0 * GB + tid);
        float xm2 = Act<T>::ld(xt + 1 * GB + tid);
        float xm1 = Act<T>::ld(xt + 2 * GB + tid);
#pragma unroll 2
        for (int j = 0; j < nst; ++j) {
          const float xv = Act<T>::ld(xt + (j + 3) * GB + tid);
          const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
          xm3 = xm2;
          xm2 = xm1;
          xm1 = xv;
          const float sc = sigmoid_f(cpre);
          const float u = cpre * sc;
          const float v = Act<T>::ld(drt + j * GB + tid) + dtb;
          const float delta = softplus_f(v);
          const float sv = sigmoid_f(v);
          const float zv = Act<T>::ld(zt + j * GB + tid);
          const float gv = Act<T>::ld(dgt + j * GB + tid);
          const float sz = sigmoid_f(zv);
          const float dy = gv * zv * sz;                           // dL/dy
          const float dzf = gv * (sz * fmaf(zv, 1.f - sz, 1.f));    // dL/dz = y * dzf
          s0[j * GB] = make_float4(delta, delta * u, dy, dzf);
          s1[j * GB] = make_float4(Dd * u, sv, sc, cpre);
        }
      }

      // ---- recompute the chunk's states from its start state ----
      {
        float2 h[NS / 2];
#pragma unroll
        for (int i = 0; i < NS / 2; ++i) {
          const int n = lane_of(i);
          h[i] = make_float2(ckt[n * GB + tid], ckt[(n + 1) * GB + tid]);
        }
#pragma unroll 2
        for (int j = 0; j < nst; ++j) {
          const float4 v0 = s0[j * GB];
          const float2 dl2 = f2b(v0.x);
          const float2 du2 = f2b(v0.y);
          const float4* B4 = reinterpret_cast<const float4*>(fB + j * NS);
#pragma unroll
          for (int qs = 0; qs < 4; ++qs) {
            const float4 bv = B4[qs ^ rot];
            const float2 dA0 = ex2x2(__fmul2_rn(dl2, a2[2 * qs]));
            const float2 dA1 = ex2x2(__fmul2_rn(dl2, a2[2 * qs + 1]));
            h[2 * qs] = __ffma2_rn(dA0, h[2 * qs], __fmul2_rn(du2, make_float2(bv.x, bv.y)));
            h[2 * qs + 1] = __ffma2_rn(dA1, h[2 * qs + 1], __fmul2_rn(du2, make_float2(bv.z, bv.w)));
          }
          tmem_st16(trow + 16u * (uint32_t)j, h);
        }
        tmem_wait_st();
      }

      // ---- reverse-time pass: y and dz, adjoint state, dA, dB/dC ----
      {
        float2 hn[NS / 2];  // h_t (state after step t)
        tmem_ld16(trow + 16u * (uint32_t)(nst - 1), hn);
#pragma unroll 2
        for (int j = nst - 1; j >= 0; --j) {
          const float4 v0 = s0[j * GB];
          const float Du = reinterpret_cast<const float*>(s1 + j * GB)[0];
          const float2 dl2 = f2b(v0.x);
          const float2 du2 = f2b(v0.y);
          const float2 dy2 = f2b(v0.z);
          float2 sB = make_float2(0.f, 0.f), sAq = make_float2(0.f, 0.f);
          float2 y01 = make_float2(0.f, 0.f), y23 = make_float2(0.f, 0.f);
          float2 pB[NS / 2], pC[NS / 2];
          float2 hp[NS / 2];  // h_{t-1}
          if (j > 0) {
            tmem_ld16(trow + 16u * (uint32_t)(j - 1), hp);
          } else {
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) {
              const int n = lane_of(i);
              hp[i] = make_float2(ckt[n * GB + tid], ckt[(n + 1) * GB + tid]);
            }
          }
          const float4* B4 = reinterpret_cast<const float4*>(fB + j * NS);
          const float4* C4 = reinterpret_cast<const float4*>(fC + j * NS);
#pragma unroll
          for (int qs = 0; qs < 4; ++qs) {
            const float4 bv = B4[qs ^ rot];
            const float4 cv = C4[qs ^ rot];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 2 * qs + e;
              const float2 bb = e ? make_float2(bv.z, bv.w) : make_float2(bv.x, bv.y);
              const float2 cc = e ? make_float2(cv.z, cv.w) : make_float2(cv.x, cv.y);
              if (e) y23 = __ffma2_rn(cc, hn[i], y23); else y01 = __ffma2_rn(cc, hn[i], y01);
              const float2 dh = __ffma2_rn(dy2, cc, carry[i]);            // dL/dh_t
              pC[i] = __fmul2_rn(dy2, hn[i]);                              // dC partial
              pB[i] = __fmul2_rn(dh, du2);                                 // dB partial
              sB = __ffma2_rn(dh, bb, sB);
              carry[i] = __fmul2_rn(ex2x2(__fmul2_rn(dl2, a2[i])), dh);    // exp(delta A) dh
              const float2 qv = __fmul2_rn(carry[i], hp[i]);               // dh exp(delta A) h_{t-1}
              dAp[i] = __ffma2_rn(dl2, qv, dAp[i]);
              sAq = __ffma2_rn(a2[i], qv, sAq);
            }
          }
#pragma unroll
          for (int i = 0; i < NS / 2; ++i) hn[i] = hp[i];
          const float y = ((y01.x + y01.y) + (y23.x + y23.y)) + Du;
          if (active) Act<T>::st(dz_c + (size_t)j * g.D, y * v0.w);
          // the scalar pass below reads these two sums
          reinterpret_cast<float*>(s0 + j * GB)[3] = sAq.x + sAq.y;
          reinterpret_cast<float*>(s1 + j * GB)[0] = sB.x + sB.y;
          // Channels past d_inner run on zero-filled inputs and parameters, so
          // their partials are exactly zero and need no masking.
          float vb[NS], vc[NS];
#pragma unroll
          for (int i = 0; i < NS / 2; ++i) {
            vb[2 * i] = pB[i].x;
            vb[2 * i + 1] = pB[i].y;
            vc[2 * i] = pC[i].x;
            vc[2 * i + 1] = pC[i].y;
          }
          const float rb = warp_sum16_rotated(vb, lane);
          const float rc = warp_sum16_rotated(vc, lane);
          const int nf = 4 * rot + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
          red[(j * NWB + warp) * 32 + (lane < 16 ? nf : 16 + nf)] = lane < 16 ? rb : rc;
        }
      }

      // ---- scalar pass: du, d delta, softplus, SiLU and conv backward ----
#pragma unroll 2
      for (int j = nst - 1; j >= 0; --j) {
        const int t = c * K + j;
        const float4 v0 = s0[j * GB];
        const float4 v1 = s1[j * GB];
        const float delta = v0.x, dy = v0.z, sAq = v0.w;
        const float sumB = v1.x, sv = v1.y, sc = v1.z, cpre = v1.w;
        const float u = cpre * sc;
        const float du = fmaf(dy, Dd, delta * sumB);
        const float ddr = fmaf(u, sumB, LN2 * sAq) * sv;
        dD_acc = fmaf(dy, u, dD_acc);
        ddtb_acc += ddr;
        if constexpr (SCAN) {  // the SiLU and conv backward run later, with du
          if (active) {
            Act<T>::st(ddr_c + (size_t)j * g.D, ddr);
            Act<T>::st(du_c + (size_t)j * g.D, du);
          }
          continue;
        }
        const float dc = du * (sc * fmaf(cpre, 1.f - sc, 1.f));
        dcb_acc += dc;
#pragma unroll
        for (int k = 0; k < WC; ++k) dcw[k] = fmaf(dc, Act<T>::ld(xt + (j + k) * GB + tid), dcw[k]);
        float dxv = fmaf(dc, w[3], fmaf(dc1, w[2], fmaf(dc2, w[1], dc3 * w[0])));
        if (ST && a.g_conv && t >= g.T - 3 && active)  // x[t] is also a conv-state output
          dxv += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + t - (g.T - 3)) * g.D + d);
        dc3 = dc2;
        dc2 = dc1;
        dc1 = dc;
        if (active) {
          Act<T>::st(ddr_c + (size_t)j * g.D, ddr);
          if (du_c) Act<T>::st(du_c + (size_t)j * g.D, du);
          if (s + 1 < g.S && t >= t_end - 3)
            a.dxpart[(((size_t)b * g.S + s) * 3 + (t - (t_end - 3))) * g.D + d] = dxv;
          else
            Act<T>::st(dx_c + (size_t)j * g.D, dxv);
          if (s > 0 && t < t_begin + 3)
            a.dchead[(((size_t)b * g.S + s) * 3 + (t - t_begin)) * g.D + d] = dc;
        }
      }
    }

    __syncthreads();
    // one global reduction per (t, n) per block for dB and dC
    for (int i = tid; i < steps * 32; i += GB) {
      const int j = i >> 5, l = i & 31;
      float v = 0.f;
#pragma unroll
      for (int ww = 0; ww < NWB; ++ww) v += red[(j * NWB + ww) * 32 + l];
      float* dst = (l < NS ? a.dB : a.dC) + ((size_t)b * g.T + c * K + j) * g.lddbc + (l & (NS - 1));
      atomicAdd(dst, v);
    }
    __syncthreads();
  }

  if (ST && s == 0 && active) {
    if (a.d_h_in) {  // carry = exp(delta_0 A) dL/dh_0 = dL/dh_{-1}
      float* dh0 = a.d_h_in + (size_t)b * NS * g.D + d;
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        const int n = lane_of(i);
        dh0[(size_t)n * g.D] = carry[i].x;
        dh0[(size_t)(n + 1) * g.D] = carry[i].y;
      }
    }
    if (!SCAN && a.d_conv_in) {
      // conv inputs of steps -1, -2, -3 reach the conv outputs of steps
      // 0..2 (dc1 = dc_0, dc2 = dc_1, dc3 = dc_2; zero past the sequence),
      // and, when T < 3, the conv-state output too
      float v[3];
      v[2] = fmaf(dc1, w[2], fmaf(dc2, w[1], dc3 * w[0]));
      v[1] = fmaf(dc1, w[1], dc2 * w[0]);
      v[0] = dc1 * w[0];
      T* dci = static_cast<T*>(a.d_conv_in) + (size_t)b * 3 * g.D + d;
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int ro = r - g.T;  // row of the conv-state output holding step r - 3
        if (a.g_conv && ro >= 0)
          v[r] += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + ro) * g.D + d);
        Act<T>::st(dci + (size_t)r * g.D, v[r]);
      }
    }
  }
  if (active) {
    float* Pp = a.partials + ((size_t)b * g.S + s) * NPART * g.D;
#pragma unroll
    for (int i = 0; i < NS / 2; ++i) {
      const int n = lane_of(i);
      Pp[(size_t)n * g.D + d] = dAp[i].x;
      Pp[(size_t)(n + 1) * g.D + d] = dAp[i].y;
    }
    Pp[(size_t)16 * g.D + d] = dD_acc;
    Pp[(size_t)17 * g.D + d] = ddtb_acc;
    Pp[(size_t)18 * g.D + d] = dcb_acc;
#pragma unroll
    for (int k = 0; k < WC; ++k) Pp[(size_t)(19 + k) * g.D + d] = dcw[k];
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_slot, a.tcols);
}

// ---------------------------------------------------------------------------
// backward main kernel with the lanes split over G = N / 8 threads per
// channel (8 lanes each, 128 / G channels per block); the threads of a
// channel take the per-step scalar work of every G-th step.  For d_state 32
// and 64, and for d_state-16 grids that fill less than one wave (each thread
// then runs about half the per-step instructions of m3_bwd_kernel and a
// block holds twice the warps per channel).  Same results as m3_bwd_kernel
// up to the order of f32 sums.
// ---------------------------------------------------------------------------

// Sum over the channels of a warp (the lanes with the same lane % G) of 8
// values held as 4 pairs, pair P holding this thread's lane pair
// P ^ ((lane >> 3) & 3).  The channel bits of a lane are its bits log2(G)
// and up; the sum runs over them:
//   G = 2: returns (in .x) the total for pair (lane >> 3) & 3, element
//          (lane >> 2) & 1 (lanes differing only in bit 1 return the same);
//   G = 4: the same total, every lane distinct;
//   G = 8: returns both elements of pair (lane >> 3) & 3.
template <int G>
__device__ __forceinline__ float2 warp_sum8_rotated(float2 (&v)[4], int lane) {
  v[0].x += __shfl_xor_sync(0xffffffffu, v[2].x, 16);
  v[0].y += __shfl_xor_sync(0xffffffffu, v[2].y, 16);
  v[1].x += __shfl_xor_sync(0xffffffffu, v[3].x, 16);
  v[1].y += __shfl_xor_sync(0xffffffffu, v[3].y, 16);
  v[0].x += __shfl_xor_sync(0xffffffffu, v[1].x, 8);
  v[0].y += __shfl_xor_sync(0xffffffffu, v[1].y, 8);
  if constexpr (G == 8) {
    return v[0];
  } else {
    const bool up = (lane & 4) != 0;
    const float send = up ? v[0].x : v[0].y;
    const float keep = up ? v[0].y : v[0].x;
    float r = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    if constexpr (G == 2) r += __shfl_xor_sync(0xffffffffu, r, 2);
    return make_float2(r, 0.f);
  }
}

template <typename T, bool ST, bool SCAN, int N>
__global__ void __launch_bounds__(128, 4) m3_bwd2_kernel(BwdArgs a) {
  constexpr int G = N / 8;     // threads per channel
  constexpr int CH = 128 / G;  // channels per block
  constexpr int NP = N + 8;    // per-channel parameter partials
  extern __shared__ __align__(128) unsigned char smem[];
  const Geo g = a.g;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int hf = tid % G;            // this thread's state lanes: 8 hf .. 8 hf + 7
  const int ch = tid / G;            // channel within the block
  const int prot = (lane >> 3) & 3;  // pair rotation for the warp reduction
  const int d0 = blockIdx.x * CH;
  const int s = blockIdx.y;
  const int b = blockIdx.z;
  const int d = d0 + ch;
  const bool active = d < g.D;
  const int c_begin = s * g.m;
  const int c_end = min(c_begin + g.m, g.nc);
  const int t_begin = c_begin * g.K;
  const int t_end = min(c_end * g.K, g.T);
  const int K = g.K;
  const Bwd2Smem L = bwd2_smem(K, sizeof(T), N);
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* dcs = reinterpret_cast<float*>(smem + L.dcs);  // [K + 3][CH]
  // state lane of register pair P
  auto lane_of = [&](int P) { return 8 * hf + 2 * (P ^ prot); };

  // recomputed states of a chunk: row j of this thread = TMEM columns
  // [8 j, 8 j + 8) of its lane; warp 0 allocates, every exit deallocates
  __shared__ uint32_t tmem_slot;
  if (warp == 0) tmem_alloc(&tmem_slot, a.tcols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t trow = tmem_slot + ((uint32_t)(warp * 32) << 16);

  float2 a2[4];
  float w[WC];
  float cb = 0.f, dtb = 0.f, Dd = 0.f;
#pragma unroll
  for (int P = 0; P < 4; ++P) {
    const int n = lane_of(P);
    a2[P].x = active ? -expf(a.a_log[(size_t)d * N + n]) * LOG2E : 0.f;
    a2[P].y = active ? -expf(a.a_log[(size_t)d * N + n + 1]) * LOG2E : 0.f;
  }
#pragma unroll
  for (int k = 0; k < WC; ++k) w[k] = active ? a.conv_w[(size_t)d * WC + k] : 0.f;
  if (active) {
    cb = a.conv_b[d];
    dtb = a.dt_bias[d];
    Dd = a.Dp[d];
  }
  float2 carry[4];
#pragma unroll
  for (int P = 0; P < 4; ++P) carry[P] = make_float2(0.f, 0.f);
  if (ST && a.g_h && active) {
    const float* gh = a.g_h + (size_t)b * N * g.D + d;
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      const int n = lane_of(P);
      carry[P] = make_float2(gh[(size_t)n * g.D], gh[(size_t)(n + 1) * g.D]);
    }
  }
  const T* xg = static_cast<const T*>(a.x);
  auto stage = [&](int c, int buf) {
    unsigned char* base = smem + (size_t)buf * L.tile;
    const int t0 = c * K;
    stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.x), xg, b, t0 - 3, K + 3, g.T, g.T, g.D, d0, tid);
    stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.dr), static_cast<const T*>(a.dr), b, t0, K, g.T, g.T, g.D, d0, tid);
    stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.z), static_cast<const T*>(a.z), b, t0, K, g.T, g.T, g.D, d0, tid);
    stage_rows<T, CH, 128>(reinterpret_cast<T*>(base + L.dg), static_cast<const T*>(a.dg), b, t0, K, g.T, g.T, g.D, d0, tid);
    stage_bc<T, 128, N>(reinterpret_cast<T*>(base + L.Bt), static_cast<const T*>(a.Bm), b, t0, K, g.T, g.T, g.ldbc, tid);
    stage_bc<T, 128, N>(reinterpret_cast<T*>(base + L.Ct), static_cast<const T*>(a.Cm), b, t0, K, g.T, g.T, g.ldbc, tid);
    stage_rows<float, CH, 128>(reinterpret_cast<float*>(base + L.ck), a.ckpt + ((size_t)b * g.nc + c) * N * g.D,
                               0, 0, N, N, N, g.D, d0, tid);
    cp_async_commit();
  };
  stage(c_end - 1, 0);
  grid_dep_trigger();
  grid_dep_wait();
  if (s + 1 < g.S) {
    const float* __restrict__ sd = a.sd;
    const float* __restrict__ q = a.q;
#pragma unroll 2
    for (int sp = g.S - 1; sp > s; --sp) {
      const size_t bs = (size_t)b * g.S + sp;
      const float2 dl2 = f2b(active ? sd[bs * g.D + d] : 0.f);
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const float* qq = q + (bs * N + lane_of(P)) * g.D + d;
        const float2 loc = active ? make_float2(qq[0], qq[g.D]) : make_float2(0.f, 0.f);
        carry[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), carry[P], loc);
      }
    }
  }
  float2 dAp[4];
#pragma unroll
  for (int P = 0; P < 4; ++P) dAp[P] = make_float2(0.f, 0.f);
  float dD_acc = 0.f, ddtb_acc = 0.f, dcb_acc = 0.f;
  float dcw[WC] = {0.f, 0.f, 0.f, 0.f};
  for (int i = tid; i < (K + 3) * CH; i += 128) dcs[i] = 0.f;  // ordered by the loop's first barrier

  for (int c = c_end - 1; c >= c_begin; --c) {
    const int buf = (c_end - 1 - c) & 1;
    if (c - 1 >= c_begin) {
      stage(c - 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const unsigned char* base = smem + (size_t)buf * L.tile;
    if (ST && a.conv_in && c * K < 3 && active && hf == 0) {
      T* xw = reinterpret_cast<T*>(smem + (size_t)buf * L.tile + L.x);
      const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * g.D + d;
      for (int r = 0; r < 3 - c * K; ++r) xw[r * CH + ch] = ci[(size_t)(c * K + r) * g.D];
    }
    {
      const T* Bt = reinterpret_cast<const T*>(base + L.Bt);
      const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
      for (int i = tid; i < K * N; i += 128) {
        fB[i] = Act<T>::ld(Bt + i);
        fC[i] = Act<T>::ld(Ct + i);
      }
    }
    __syncthreads();
    const T* xt = reinterpret_cast<const T*>(base + L.x);  // row r is step c*K - 3 + r
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const T* dgt = reinterpret_cast<const T*>(base + L.dg);
    const float* ckt = reinterpret_cast<const float*>(base + L.ck);
    const int steps = min(K, g.T - c * K);
    float4* s0 = reinterpret_cast<float4*>(smem + L.scal) + ch;  // shared by the channel's threads, stride CH
    float4* s1 = s0 + (size_t)K * CH;
    const size_t row0 = ((size_t)b * g.T + (size_t)c * K) * g.D + d;

    // ---- scalar pass, every G-th step ----
    for (int j = hf; j < steps; j += G) {
      const float xm3 = Act<T>::ld(xt + j * CH + ch);
      const float xm2 = Act<T>::ld(xt + (j + 1) * CH + ch);
      const float xm1 = Act<T>::ld(xt + (j + 2) * CH + ch);
      const float xv = Act<T>::ld(xt + (j + 3) * CH + ch);
      const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
      const float sc = sigmoid_f(cpre);
      const float u = cpre * sc;
      const float v = Act<T>::ld(drt + j * CH + ch) + dtb;
      const float delta = softplus_f(v);
      const float sv = sigmoid_f(v);
      const float zv = Act<T>::ld(zt + j * CH + ch);
      const float gv = Act<T>::ld(dgt + j * CH + ch);
      const float sz = sigmoid_f(zv);
      s0[j * CH] = make_float4(delta, delta * u, gv * zv * sz, gv * (sz * fmaf(zv, 1.f - sz, 1.f)));
      s1[j * CH] = make_float4(Dd * u, sv, sc, cpre);
    }
    __syncwarp();

    // ---- recompute this thread's 8 lanes of the chunk's states ----
    {
      float2 h[4];
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const int n = lane_of(P);
        h[P] = make_float2(ckt[n * CH + ch], ckt[(n + 1) * CH + ch]);
      }
#pragma unroll 2
      for (int j = 0; j < steps; ++j) {
        const float4 v0 = s0[j * CH];
        const float2 dl2 = f2b(v0.x);
        const float2 du2 = f2b(v0.y);
#pragma unroll
        for (int P = 0; P < 4; ++P) {
          const float2 bb = *reinterpret_cast<const float2*>(fB + j * N + lane_of(P));
          h[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), h[P], __fmul2_rn(du2, bb));
        }
        tmem_st8(trow + 8u * (uint32_t)j, h);
      }
      tmem_wait_st();
    }

    // ---- reverse-time pass ----
    {
      float2 hn[4];
      tmem_ld8(trow + 8u * (uint32_t)(steps - 1), hn);
#pragma unroll 2
      for (int j = steps - 1; j >= 0; --j) {
        const float4 v0 = s0[j * CH];
        const float Du = reinterpret_cast<const float*>(s1 + j * CH)[0];
        const float2 dl2 = f2b(v0.x);
        const float2 du2 = f2b(v0.y);
        const float2 dy2 = f2b(v0.z);
        float2 sB = make_float2(0.f, 0.f), sAq = make_float2(0.f, 0.f), y2 = make_float2(0.f, 0.f);
        float2 pB[4], pC[4], hp[4];
        if (j > 0) {
          tmem_ld8(trow + 8u * (uint32_t)(j - 1), hp);
        } else {
#pragma unroll
          for (int P = 0; P < 4; ++P) {
            const int n = lane_of(P);
            hp[P] = make_float2(ckt[n * CH + ch], ckt[(n + 1) * CH + ch]);
          }
        }
#pragma unroll
        for (int P = 0; P < 4; ++P) {
          const float2 bb = *reinterpret_cast<const float2*>(fB + j * N + lane_of(P));
          const float2 cc = *reinterpret_cast<const float2*>(fC + j * N + lane_of(P));
          y2 = __ffma2_rn(cc, hn[P], y2);
          const float2 dh = __ffma2_rn(dy2, cc, carry[P]);
          pC[P] = __fmul2_rn(dy2, hn[P]);
          pB[P] = __fmul2_rn(dh, du2);
          sB = __ffma2_rn(dh, bb, sB);
          carry[P] = __fmul2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), dh);
          const float2 qv = __fmul2_rn(carry[P], hp[P]);
          dAp[P] = __ffma2_rn(dl2, qv, dAp[P]);
          sAq = __ffma2_rn(a2[P], qv, sAq);
        }
#pragma unroll
        for (int P = 0; P < 4; ++P) hn[P] = hp[P];
        float ys = y2.x + y2.y, sBs = sB.x + sB.y, sAs = sAq.x + sAq.y;
#pragma unroll
        for (int o = 1; o < G; o <<= 1) {
          ys += __shfl_xor_sync(0xffffffffu, ys, o);
          sBs += __shfl_xor_sync(0xffffffffu, sBs, o);
          sAs += __shfl_xor_sync(0xffffffffu, sAs, o);
        }
        if (hf == j % G) {
          if (active) Act<T>::st(static_cast<T*>(a.dz) + row0 + (size_t)j * g.D, (ys + Du) * v0.w);
          reinterpret_cast<float*>(s0 + j * CH)[3] = sAs;
          reinterpret_cast<float*>(s1 + j * CH)[0] = sBs;
        }
        const float2 rb = warp_sum8_rotated<G>(pB, lane);
        const float2 rc = warp_sum8_rotated<G>(pC, lane);
        float* rj = red + (j * 4 + warp) * 2 * N;  // [dB: N][dC: N]
        if constexpr (G == 8) {
          const int n = 8 * hf + 2 * prot;
          rj[n] = rb.x;
          rj[n + 1] = rb.y;
          rj[N + n] = rc.x;
          rj[N + n + 1] = rc.y;
        } else if (G == 4 || (lane & 2) == 0) {
          const int n = 8 * hf + 2 * prot + ((lane >> 2) & 1);
          rj[n] = rb.x;
          rj[N + n] = rc.x;
        }
      }
    }
    __syncwarp();

    // ---- du, d delta, softplus and (unless SCAN) SiLU backward, every G-th step ----
    for (int j = hf; j < steps; j += G) {
      const int t = c * K + j;
      const float4 v0 = s0[j * CH];
      const float4 v1 = s1[j * CH];
      const float delta = v0.x, dy = v0.z, sAq = v0.w;
      const float sumB = v1.x, sv = v1.y, sc = v1.z, cpre = v1.w;
      const float u = cpre * sc;
      const float du = fmaf(dy, Dd, delta * sumB);
      const float ddr = fmaf(u, sumB, LN2 * sAq) * sv;
      dD_acc = fmaf(dy, u, dD_acc);
      ddtb_acc += ddr;
      if (active) {
        Act<T>::st(static_cast<T*>(a.ddr) + row0 + (size_t)j * g.D, ddr);
        if (a.du_dbg) Act<T>::st(static_cast<T*>(a.du_dbg) + row0 + (size_t)j * g.D, du);
      }
      if constexpr (SCAN) continue;
      const float dc = du * (sc * fmaf(cpre, 1.f - sc, 1.f));
      dcb_acc += dc;
#pragma unroll
      for (int k = 0; k < WC; ++k) dcw[k] = fmaf(dc, Act<T>::ld(xt + (j + k) * CH + ch), dcw[k]);
      dcs[j * CH + ch] = dc;
      if (active && s > 0 && t < t_begin + 3)
        a.dchead[(((size_t)b * g.S + s) * 3 + (t - t_begin)) * g.D + d] = dc;
    }
    if constexpr (!SCAN) {
      __syncwarp();
      // ---- conv backward: d_x from the conv-input gradient of this and the next 3 steps ----
      for (int j = hf; j < steps; j += G) {
        const int t = c * K + j;
        float dxv = fmaf(dcs[j * CH + ch], w[3], fmaf(dcs[(j + 1) * CH + ch], w[2],
                         fmaf(dcs[(j + 2) * CH + ch], w[1], dcs[(j + 3) * CH + ch] * w[0])));
        if (ST && a.g_conv && t >= g.T - 3 && active)
          dxv += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + t - (g.T - 3)) * g.D + d);
        if (active) {
          if (s + 1 < g.S && t >= t_end - 3)
            a.dxpart[(((size_t)b * g.S + s) * 3 + (t - (t_end - 3))) * g.D + d] = dxv;
          else
            Act<T>::st(static_cast<T*>(a.dx) + row0 + (size_t)j * g.D, dxv);
        }
      }
      __syncwarp();
      // the next chunk processed (the one before in time) reads the dc of
      // this chunk's first three steps: rows 0..2 of this chunk followed by
      // the carried rows (a chunk may be shorter than three steps), all
      // read before any is overwritten
      if (hf == 0) {
        const float v0 = dcs[ch], v1 = dcs[CH + ch], v2 = dcs[2 * CH + ch];
        dcs[K * CH + ch] = v0;
        dcs[(K + 1) * CH + ch] = v1;
        dcs[(K + 2) * CH + ch] = v2;
      }
    }

    __syncthreads();
    for (int i = tid; i < steps * 2 * N; i += 128) {
      const int j = i / (2 * N), l = i % (2 * N);
      float v = 0.f;
#pragma unroll
      for (int ww = 0; ww < 4; ++ww) v += red[(j * 4 + ww) * 2 * N + l];
      float* dst = (l < N ? a.dB : a.dC) + ((size_t)b * g.T + c * K + j) * g.lddbc + (l & (N - 1));
      atomicAdd(dst, v);
    }
    __syncthreads();
  }

  if (ST && s == 0 && active) {
    if (a.d_h_in) {
      float* dh0 = a.d_h_in + (size_t)b * N * g.D + d;
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const int n = lane_of(P);
        dh0[(size_t)n * g.D] = carry[P].x;
        dh0[(size_t)(n + 1) * g.D] = carry[P].y;
      }
    }
    if (!SCAN && a.d_conv_in && hf == 0) {
      // dc of steps 0, 1, 2 (zero past the sequence), kept in rows K.. K+2
      const float f0 = dcs[K * CH + ch], f1 = dcs[(K + 1) * CH + ch], f2 = dcs[(K + 2) * CH + ch];
      float v[3];
      v[2] = fmaf(f0, w[2], fmaf(f1, w[1], f2 * w[0]));
      v[1] = fmaf(f0, w[1], f1 * w[0]);
      v[0] = f0 * w[0];
      T* dci = static_cast<T*>(a.d_conv_in) + (size_t)b * 3 * g.D + d;
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int ro = r - g.T;
        if (a.g_conv && ro >= 0)
          v[r] += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + ro) * g.D + d);
        Act<T>::st(dci + (size_t)r * g.D, v[r]);
      }
    }
  }
  // the per-step partial sums: each thread of a channel summed its own steps
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, o);
    ddtb_acc += __shfl_xor_sync(0xffffffffu, ddtb_acc, o);
    dcb_acc += __shfl_xor_sync(0xffffffffu, dcb_acc, o);
#pragma unroll
    for (int k = 0; k < WC; ++k) dcw[k] += __shfl_xor_sync(0xffffffffu, dcw[k], o);
  }
  if (active) {
    float* Pp = a.partials + ((size_t)b * g.S + s) * NP * g.D;
#pragma unroll
    for (int P = 0; P < 4; ++P) {
      const int n = lane_of(P);
      Pp[(size_t)n * g.D + d] = dAp[P].x;
      Pp[(size_t)(n + 1) * g.D + d] = dAp[P].y;
    }
    if (hf == 0) {
      Pp[(size_t)N * g.D + d] = dD_acc;
      Pp[(size_t)(N + 1) * g.D + d] = ddtb_acc;
      Pp[(size_t)(N + 2) * g.D + d] = dcb_acc;
#pragma unroll
      for (int k = 0; k < WC; ++k) Pp[(size_t)(N + 3 + k) * g.D + d] = dcw[k];
    }
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_slot, a.tcols);
}

// The backward's last kernel, two roles by block index.
//  - blocks [0, nfin): parameter gradients, the per-(batch, segment) partials
//    summed in a fixed order (32 outputs per block, rows split over its 8
//    warps and combined in a fixed tree), so the result is deterministic;
//  - blocks [nfin, ...): d_x at the last three steps of each segment but the
//    last, which needs the conv gradient of the next segment's first steps.
// N = d_state: partial rows per channel are N + 8 (N of dA, then dD,
// d_dt_bias, d_conv_b, d_conv_w[0..3]); nout of them are finalized.
template <typename T>
__global__ void m3_bwd_tail_kernel(BwdArgs a, int rows, int nfin, int nout, int N) {
  const Geo g = a.g;
  grid_dep_wait();  // the main kernel's partials and boundary terms
  if ((int)blockIdx.x >= nfin) {
    const size_t idx = (size_t)(blockIdx.x - nfin) * blockDim.x + threadIdx.x;
    const size_t total = (size_t)g.B * (g.S - 1) * 3 * g.D;
    if (idx >= total) return;
    const int d = (int)(idx % g.D);
    size_t rest = idx / g.D;
    const int j = (int)(rest % 3);
    rest /= 3;
    const int s = (int)(rest % (g.S - 1));
    const int b = (int)(rest / (g.S - 1));
    const int t_end = min((s + 1) * g.m * g.K, g.T);
    const int t = t_end - 3 + j;
    float v = a.dxpart[(((size_t)b * g.S + s) * 3 + j) * g.D + d];
    for (int k = 0; k < WC; ++k) {
      const int tp = t + 3 - k;
      if (tp >= t_end && tp < g.T)
        v = fmaf(a.dchead[(((size_t)b * g.S + s + 1) * 3 + (tp - t_end)) * g.D + d],
                 a.conv_w[(size_t)d * WC + k], v);
    }
    Act<T>::st(static_cast<T*>(a.dx) + ((size_t)b * g.T + t) * g.D + d, v);
    return;
  }
  // 32 consecutive outputs per block (coalesced row reads), rows split over
  // the block's 8 warps: warp w sums rows w, w + 8, ... in order, then warp
  // 0 adds the 8 partial sums in a fixed order.
  __shared__ float part[8][33];
  const int cx = threadIdx.x & 31, ry = threadIdx.x >> 5;
  const int oidx = blockIdx.x * 32 + cx;
  const bool ok = oidx < nout * g.D;
  const int jj = oidx / g.D, d = oidx - jj * g.D;
  {
    float v0 = 0.f, v1 = 0.f;
    if (ok) {
      const float* __restrict__ P = a.partials + (size_t)jj * g.D + d;
      const size_t stride = (size_t)(N + 8) * g.D;
      int r = ry;
#pragma unroll 4
      for (; r + 8 < rows; r += 16) {
        v0 += P[(size_t)r * stride];
        v1 += P[(size_t)(r + 8) * stride];
      }
      if (r < rows) v0 += P[(size_t)r * stride];
    }
    part[ry][cx] = v0 + v1;
  }
  __syncthreads();
  if (ry != 0 || !ok) return;
  float v = ((part[0][cx] + part[1][cx]) + (part[2][cx] + part[3][cx])) +
            ((part[4][cx] + part[5][cx]) + (part[6][cx] + part[7][cx]));
  float* dst;
  if (jj < N) {
    v *= -expf(a.a_log[(size_t)d * N + jj]);  // dL/da_log = dL/dA * A
    dst = a.d_a_log + (size_t)d * N + jj;
  } else if (jj == N) {
    dst = a.dD + d;
  } else if (jj == N + 1) {
    dst = a.d_dt_bias + d;
  } else if (jj == N + 2) {
    dst = a.d_conv_b + d;
  } else {
    dst = a.d_conv_w + (size_t)d * WC + (jj - N - 3);
  }
  *dst = a.accumulate ? *dst + v : v;
}

// ---------------------------------------------------------------------------
// SiLU and conv backward of the two-phase backward: with du from the scan
// backward and a gradient reaching u from outside the layer core (the x_proj
// path), dc = (du + du_extra) silu'(c) and d_x[s] = sum_k dc[s+3-k] w[k];
// per-(batch, tile) partials of d_conv_b and d_conv_w.  One thread per
// channel over a tile of steps, plus the three steps after it, whose dc
// reaches the tile's last d_x.  Plain coalesced loads: every value is read
// by one thread.
// ---------------------------------------------------------------------------

struct ConvArgs {
  int B, T, D, tile, ntiles;
  const void *x, *du, *du_extra;  // [B, T, D] act (du_extra nullable)
  const float *conv_w, *conv_b;
  void* dx;                       // [B, T, D] act
  float* part;                    // [B * ntiles, 5, D]: d_conv_b, d_conv_w[0..3]
  const void* conv_in;            // [B, 3, D] act, nullable
  const void* g_conv;             // [B, 3, D] act, nullable
  void* d_conv_in;                // [B, 3, D] act, nullable
  float *d_conv_w, *d_conv_b;
  int accumulate;
};

// Steps per conv-backward tile: rows [t0 - 3, t0 + CT + 3) of x and
// [t0, t0 + CT + 3) of du and du_extra are staged in shared memory by 16-byte
// copies, so each thread's walk over the tile reads no global memory.
constexpr int CT = 32;
struct ConvSmem {
  size_t x, du, de, total;
};
__host__ __device__ inline ConvSmem conv_smem(int es) {
  ConvSmem s;
  s.x = 0;
  s.du = align_up((size_t)(CT + 6) * 128 * es, 128);
  s.de = s.du + align_up((size_t)(CT + 3) * 128 * es, 128);
  s.total = s.de + align_up((size_t)(CT + 3) * 128 * es, 128);
  return s;
}

template <typename T>
__global__ void __launch_bounds__(128) m3_conv_bwd_kernel(ConvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int d0 = blockIdx.x * 128;
  const int d = d0 + tid;
  const int tile = blockIdx.y, b = blockIdx.z;
  const size_t D = (size_t)a.D;
  const int t0 = tile * CT;
  const int t1 = min(t0 + CT, a.T);
  const ConvSmem L = conv_smem(sizeof(T));
  T* xs = reinterpret_cast<T*>(smem + L.x);    // row r: step t0 - 3 + r
  T* us = reinterpret_cast<T*>(smem + L.du);   // row r: step t0 + r
  T* es = reinterpret_cast<T*>(smem + L.de);
  stage_rows<T, 128, 128>(xs, static_cast<const T*>(a.x), b, t0 - 3, CT + 6, a.T, a.T, a.D, d0, tid);
  stage_rows<T, 128, 128>(us, static_cast<const T*>(a.du), b, t0, CT + 3, a.T, a.T, a.D, d0, tid);
  if (a.du_extra)
    stage_rows<T, 128, 128>(es, static_cast<const T*>(a.du_extra), b, t0, CT + 3, a.T, a.T, a.D, d0, tid);
  cp_async_commit();
  const bool active = d < a.D;
  float w[WC] = {0.f, 0.f, 0.f, 0.f};
  float cb = 0.f;
  if (active) {
#pragma unroll
    for (int k = 0; k < WC; ++k) w[k] = a.conv_w[(size_t)d * WC + k];
    cb = a.conv_b[d];
  }
  cp_async_wait<0>();
  __syncthreads();
  if (!active) return;  // no barriers below
  if (a.conv_in && t0 < 3) {
    // halo rows before step 0 (staged as zeros): the carried conv inputs
    const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * D + d;
    for (int r = 0; r < 3 - t0; ++r) xs[r * 128 + tid] = ci[(size_t)(t0 + r) * D];
  }
  // dc of steps t0 .. t1 + 2 (zero from step T on), then d_x of the tile
  float dcs[CT + 3];
  float dcb = 0.f, dcw[WC] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < CT + 3; ++j) {
    const int t = t0 + j;
    float dc = 0.f;
    if (t < a.T) {
      const float xm3 = Act<T>::ld(xs + j * 128 + tid);
      const float xm2 = Act<T>::ld(xs + (j + 1) * 128 + tid);
      const float xm1 = Act<T>::ld(xs + (j + 2) * 128 + tid);
      const float xv = Act<T>::ld(xs + (j + 3) * 128 + tid);
      float gu = Act<T>::ld(us + j * 128 + tid);
      if (a.du_extra) gu += Act<T>::ld(es + j * 128 + tid);
      const float c = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
      const float sc = sigmoid_f(c);
      dc = gu * (sc * fmaf(c, 1.f - sc, 1.f));
      if (j < CT && t < t1) {
        dcb += dc;
        dcw[0] = fmaf(dc, xm3, dcw[0]);
        dcw[1] = fmaf(dc, xm2, dcw[1]);
        dcw[2] = fmaf(dc, xm1, dcw[2]);
        dcw[3] = fmaf(dc, xv, dcw[3]);
      }
    }
    dcs[j] = dc;
  }
#pragma unroll
  for (int j = 0; j < CT; ++j) {
    const int t = t0 + j;
    if (t < t1) {
      float v = fmaf(dcs[j], w[3], fmaf(dcs[j + 1], w[2], fmaf(dcs[j + 2], w[1], dcs[j + 3] * w[0])));
      if (a.g_conv && t >= a.T - 3)  // x[t] is also a conv-state output
        v += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + t - (a.T - 3)) * D + d);
      Act<T>::st(static_cast<T*>(a.dx) + ((size_t)b * a.T + t) * D + d, v);
    }
  }
  if (tile == 0 && a.d_conv_in) {
    // conv inputs of steps -3, -2, -1 (rows 0..2) reach dc of steps 0..2
    float v[3];
    v[0] = dcs[0] * w[0];
    v[1] = fmaf(dcs[1], w[0], dcs[0] * w[1]);
    v[2] = fmaf(dcs[2], w[0], fmaf(dcs[1], w[1], dcs[0] * w[2]));
    T* dci = static_cast<T*>(a.d_conv_in) + (size_t)b * 3 * D + d;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const int ro = r - a.T;  // row of the conv-state output holding step r - 3
      if (a.g_conv && ro >= 0)
        v[r] += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + ro) * D + d);
      Act<T>::st(dci + (size_t)r * D, v[r]);
    }
  }
  float* P = a.part + ((size_t)b * a.ntiles + tile) * 5 * D + d;
  P[0] = dcb;
#pragma unroll
  for (int k = 0; k < WC; ++k) P[(size_t)(1 + k) * D] = dcw[k];
}

// d_conv_b and d_conv_w from the per-(batch, tile) partials, summed in a
// fixed order (32 outputs per block, rows split over 8 warps).
__global__ void m3_conv_fin_kernel(ConvArgs a) {
  grid_dep_wait();  // the conv backward's partials
  __shared__ float part[8][33];
  const int cx = threadIdx.x & 31, ry = threadIdx.x >> 5;
  const int oidx = blockIdx.x * 32 + cx;
  const bool ok = oidx < 5 * a.D;
  const int j = ok ? oidx / a.D : 0, d = oidx - j * a.D;
  const int rows = a.B * a.ntiles;
  float v0 = 0.f;
  if (ok) {
    const float* __restrict__ P = a.part + (size_t)j * a.D + d;
    const size_t stride = (size_t)5 * a.D;
    float v1 = 0.f;
    int r = ry;
#pragma unroll 4
    for (; r + 8 < rows; r += 16) {
      v0 += P[(size_t)r * stride];
      v1 += P[(size_t)(r + 8) * stride];
    }
    if (r < rows) v0 += P[(size_t)r * stride];
    v0 += v1;
  }
  part[ry][cx] = v0;
  __syncthreads();
  if (ry != 0 || !ok) return;
  const float v = ((part[0][cx] + part[1][cx]) + (part[2][cx] + part[3][cx])) +
                  ((part[4][cx] + part[5][cx]) + (part[6][cx] + part[7][cx]));
  float* dst = j == 0 ? a.d_conv_b + d : a.d_conv_w + (size_t)d * WC + (j - 1);
  *dst = a.accumulate ? *dst + v : v;
}

// ---------------------------------------------------------------------------
// decode: the forward of a short window (typically one token per sequence)
// from the carried state, updating that state in place; no checkpoints, no
// time split.  One thread per channel keeps its N state lanes in registers;
// B_t and C_t of each step are staged in shared memory for the block.
// ---------------------------------------------------------------------------

struct DecArgs {
  int B, T, D;
  int ldbc;  // row stride (elements) of Bm and Cm
  const void *x, *dr, *z, *Bm, *Cm;
  const float *conv_w, *conv_b, *dt_bias, *a_log, *Dp;
  float* h;    // [B, N, D] f32, in and out
  void* conv;  // [B, 3, D] act, in and out
  void *gated, *y_dbg;
};

constexpr int GD = 128;  // decode: channels (= threads) per block

// Each channel's N lanes are split over G = N / 16 neighbouring threads of
// a warp (16 lanes each; y is summed over the G threads with shuffles), so
// every d_state keeps 16 state lanes per thread.  R batch rows per thread
// (two when the grid is large enough) keep more loads in flight.  Each step
// issues all of its global loads before its barrier; B and C of the next
// step are staged into the other half of a double buffer.
template <typename T, int N, int R>
__global__ void __launch_bounds__(GD) m3_decode_kernel(DecArgs a) {
  constexpr int G = N / 16;       // threads per channel
  constexpr int CH = GD / G;      // channels per block
  constexpr int NB = 2 * N * R;   // B and C values of one step
  __shared__ float sBC[2][R][2 * N];
  __shared__ float sA[8][GD][2];  // A log2(e) of this thread's lanes
  const int tid = threadIdx.x;
  const int q = tid % G;          // this thread's lanes: 16 q .. 16 q + 15
  const int d = blockIdx.x * CH + tid / G;
  const bool active = d < a.D;
  const size_t D = (size_t)a.D;
  int rb[R];
  bool ron[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    rb[r] = blockIdx.y * R + r;
    ron[r] = active && rb[r] < a.B;
  }
  auto stage = [&](int t, int buf) {
    for (int i = tid; i < NB; i += GD) {
      const int sr = i / (2 * N), sn = i % (2 * N);
      const int sb = blockIdx.y * R + sr;
      if (sb < a.B) {
        const T* src = static_cast<const T*>(sn < N ? a.Bm : a.Cm);
        sBC[buf][sr][sn] = Act<T>::ld(src + ((size_t)sb * a.T + t) * a.ldbc + (sn & (N - 1)));
      }
    }
  };
  if (a.T > 0) stage(0, 0);

  float2 h[R][8];
  float w[WC] = {0.f, 0.f, 0.f, 0.f};
  float xm3[R], xm2[R], xm1[R];
  float cb = 0.f, dtb = 0.f, Dd = 0.f;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    xm3[r] = xm2[r] = xm1[r] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) h[r][i] = make_float2(0.f, 0.f);
  }
  // every load of the first step is issued before the first use of any
  float xn[R], dn[R], zn[R];  // x, delta_raw, z of the next step
  auto prefetch = [&](int t) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      xn[r] = dn[r] = zn[r] = 0.f;
      if (ron[r]) {
        const size_t i = ((size_t)rb[r] * a.T + t) * D + d;
        xn[r] = Act<T>::ld(static_cast<const T*>(a.x) + i);
        dn[r] = Act<T>::ld(static_cast<const T*>(a.dr) + i);
        zn[r] = Act<T>::ld(static_cast<const T*>(a.z) + i);
      }
    }
  };
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!ron[r]) continue;
    const float* hp = a.h + ((size_t)rb[r] * N + 16 * q) * D + d;
#pragma unroll
    for (int i = 0; i < 8; ++i) h[r][i] = make_float2(hp[(size_t)(2 * i) * D], hp[(size_t)(2 * i + 1) * D]);
    const T* cp = static_cast<const T*>(a.conv) + (size_t)rb[r] * 3 * D + d;
    xm3[r] = Act<T>::ld(cp);
    xm2[r] = Act<T>::ld(cp + D);
    xm1[r] = Act<T>::ld(cp + 2 * D);
  }
  if (a.T > 0) prefetch(0);
  if (active) {
#pragma unroll
    for (int k = 0; k < WC; ++k) w[k] = a.conv_w[(size_t)d * WC + k];
    cb = a.conv_b[d];
    dtb = a.dt_bias[d];
    Dd = a.Dp[d];
    const float* al = a.a_log + (size_t)d * N + 16 * q;  // 4-byte aligned only
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sA[i][tid][0] = -expf(al[2 * i]) * LOG2E;
      sA[i][tid][1] = -expf(al[2 * i + 1]) * LOG2E;
    }
  }

#pragma unroll 1
  for (int t = 0; t < a.T; ++t) {
    float xv[R], dr[R], zv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      xv[r] = xn[r];
      dr[r] = dn[r];
      zv[r] = zn[r];
    }
    if (t + 1 < a.T) {
      prefetch(t + 1);
      stage(t + 1, (t + 1) & 1);
    }
    __syncthreads();  // step t's B and C (and, at t = 0, A) are visible
    const int buf = t & 1;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float cpre = fmaf(w[0], xm3[r], fmaf(w[1], xm2[r], fmaf(w[2], xm1[r], fmaf(w[3], xv[r], cb))));
      xm3[r] = xm2[r];
      xm2[r] = xm1[r];
      xm1[r] = xv[r];
      const float u = cpre * sigmoid_f(cpre);
      const float delta = softplus_f(dr[r] + dtb);
      const float2 dl2 = f2b(delta);
      const float2 du2 = f2b(delta * u);
      float2 y2 = make_float2(0.f, 0.f);
      const float* bc = sBC[buf][r] + 16 * q;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 bb = *reinterpret_cast<const float2*>(bc + 2 * k);
        const float2 cc = *reinterpret_cast<const float2*>(bc + N + 2 * k);
        const float2 a2 = *reinterpret_cast<const float2*>(sA[k][tid]);
        h[r][k] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2)), h[r][k], __fmul2_rn(du2, bb));
        y2 = __ffma2_rn(cc, h[r][k], y2);
      }
      float ys = y2.x + y2.y;
#pragma unroll
      for (int o = 1; o < G; o <<= 1) ys += __shfl_xor_sync(0xffffffffu, ys, o);
      if (ron[r] && q == 0) {
        const size_t i = ((size_t)rb[r] * a.T + t) * D + d;
        const float y = ys + Dd * u;
        Act<T>::st(static_cast<T*>(a.gated) + i, y * (zv[r] * sigmoid_f(zv[r])));
        if (a.y_dbg) Act<T>::st(static_cast<T*>(a.y_dbg) + i, y);
      }
    }
    __syncthreads();  // step t's buffer is free for step t + 2
  }
  if (a.T == 0) return;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!ron[r]) continue;
    float* hp = a.h + ((size_t)rb[r] * N + 16 * q) * D + d;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      hp[(size_t)(2 * i) * D] = h[r][i].x;
      hp[(size_t)(2 * i + 1) * D] = h[r][i].y;
    }
    if (q == 0) {
      T* cp = static_cast<T*>(a.conv) + (size_t)rb[r] * 3 * D + d;
      Act<T>::st(cp, xm3[r]);
      Act<T>::st(cp + D, xm2[r]);
      Act<T>::st(cp + 2 * D, xm1[r]);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// opt-in shared memory per block, less 1 KB kept for static shared memory
constexpr size_t SMEM_CAP = 227 * 1024 - 1024;

// Tensor-memory columns a backward CTA allocates for K rows of 16 states:
// a power of two >= 32 (the allocation granularity), at most 512.
__host__ inline uint32_t tmem_cols_for(int K) {
  uint32_t c = 32;
  while (c < (uint32_t)K * NS) c <<= 1;
  return c;
}

// Tensor-memory columns of a two-thread-per-channel backward CTA: 8 per step.
__host__ inline uint32_t tmem_cols2_for(int K) {
  uint32_t c = 32;
  while (c < (uint32_t)K * 8) c <<= 1;
  return c;
}

// Largest chunk whose backward fits: 16 K tensor-memory columns <= 512 and
// the shared-memory footprint within one block's limit.
__host__ inline int kmax_for(int es) {
  int k = KMAX;
  while (k > 1 && (bwd_smem(k, es).total > SMEM_CAP || tmem_cols_for(k) > 512)) --k;
  return k;
}

// Shared memory to request per backward CTA: its footprint, raised if needed
// so that no more CTAs fit on one SM than tensor memory can serve at once
// (512 columns / tcols), so no allocation ever has to wait.
__host__ inline size_t bwd_launch_smem(int K, int es, int smem_per_sm) {
  const int max_ctas = 512 / (int)tmem_cols_for(K);
  size_t need = bwd_smem(K, es).total;
  const size_t floor_bytes = (size_t)smem_per_sm / (max_ctas + 1) + 1;  // > 1/(max+1) of the SM
  if (need < floor_bytes) need = floor_bytes;
  return align_up(need, 128);
}

// The same residency cap for the two-thread backward.
__host__ inline size_t bwd2_launch_smem(int K, int es, int N, int smem_per_sm) {
  const int max_ctas = 512 / (int)tmem_cols2_for(K);
  size_t need = bwd2_smem(K, es, N).total;
  const size_t floor_bytes = (size_t)smem_per_sm / (max_ctas + 1) + 1;
  if (need < floor_bytes) need = floor_bytes;
  return align_up(need, 128);
}

struct DevInfo {
  bool attrs = false;
  int sms = 0;
  int smem_per_sm = 0;
  int occ_fwd[2][KMAX + 1];  // [dtype][chunk] blocks per SM, 0 = not yet queried
  int occ_bwd[2][KMAX + 1];
};

std::mutex g_mu;
DevInfo g_dev[64];
thread_local cudaError_t g_last_cuda = cudaSuccess;  // last CUDA error this thread saw

// Record a failed CUDA call (and clear the runtime's sticky-free error state).
inline cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess) {
    g_last_cuda = e;
    cudaGetLastError();
  }
  return e;
}

// the split kernels for d_state N
template <typename T, bool ST, bool SCAN>
void (*bwd2_for(int N))(BwdArgs) {
  return N == 16 ? m3_bwd2_kernel<T, ST, SCAN, 16>
       : N == 32 ? m3_bwd2_kernel<T, ST, SCAN, 32> : m3_bwd2_kernel<T, ST, SCAN, 64>;
}
template <typename T>
void (*agg_for(bool split, int N))(BwdArgs) {
  if (!split) return m3_bwd_agg_kernel<T, 1, 16>;
  return N == 16 ? m3_bwd_agg_kernel<T, 2, 16>
       : N == 32 ? m3_bwd_agg_kernel<T, 4, 32> : m3_bwd_agg_kernel<T, 8, 64>;
}

template <typename T>
cudaError_t set_attrs() {
  const int es = sizeof(T);
  cudaError_t e;
  // every kernel here wants all of the unified L1/shared storage as shared
  // memory, so that the occupancy the runtime reports is the one it launches
  e = cudaFuncSetAttribute(m3_fwd_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fwd_smem(es).total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_fwd_kernel<T, true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_fwd_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)fwd_smem(es).total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_fwd_kernel<T, false>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  const bool splits[4] = {false, true, true, true};
  const int ns[4] = {16, 16, 32, 64};
  for (int i = 0; i < 4; ++i) {
    void (*k)(BwdArgs) = agg_for<T>(splits[i], ns[i]);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)agg_smem(es, ns[i]).total);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  for (int N : {16, 32, 64}) {
    void (*fk[2])(FwdArgs) = {N == 16 ? m3_fwd2_kernel<T, false, 16> : N == 32 ? m3_fwd2_kernel<T, false, 32>
                                                                                : m3_fwd2_kernel<T, false, 64>,
                              N == 16 ? m3_fwd2_kernel<T, true, 16> : N == 32 ? m3_fwd2_kernel<T, true, 32>
                                                                               : m3_fwd2_kernel<T, true, 64>};
    for (auto k : fk) {
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fwd2_smem(es, N).total);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    }
  }
  void (*const bwd_kernels[16])(BwdArgs) = {
      m3_bwd_kernel<T, false, false>, m3_bwd_kernel<T, true, false>, m3_bwd_kernel<T, false, true>,
      m3_bwd_kernel<T, true, true>,
      bwd2_for<T, false, false>(16), bwd2_for<T, true, false>(16), bwd2_for<T, false, true>(16),
      bwd2_for<T, true, true>(16),
      bwd2_for<T, false, false>(32), bwd2_for<T, true, false>(32), bwd2_for<T, false, true>(32),
      bwd2_for<T, true, true>(32),
      bwd2_for<T, false, false>(64), bwd2_for<T, true, false>(64), bwd2_for<T, false, true>(64),
      bwd2_for<T, true, true>(64)};
  for (auto k : bwd_kernels) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_CAP);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_conv_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)conv_smem(es).total);
  return e;
}

// Device facts for the current device: kernel attributes are set once per
// device (with that device current), occupancy is queried once per chunk.
cudaError_t device_info(int chunk, int ai, int* sms, int* occ_f, int* occ_b, int* smem_sm = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& di = g_dev[dev];
  if (!di.attrs) {
    e = set_attrs<float>();
    if (e != cudaSuccess) return e;
    e = set_attrs<__nv_bfloat16>();
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    for (int a = 0; a < 2; ++a)
      for (int k = 0; k <= KMAX; ++k) di.occ_fwd[a][k] = di.occ_bwd[a][k] = 0;
    di.attrs = true;
  }
  if (occ_f && di.occ_fwd[ai][chunk] == 0) {
    int of = 0, ob = 0;
    if (ai == 1) {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&of, m3_fwd_kernel<__nv_bfloat16, true>, GF,
                                                        fwd_smem(2).total);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ob, m3_bwd_kernel<__nv_bfloat16, false, false>, GB,
                                                          bwd_launch_smem(chunk, 2, di.smem_per_sm));
    } else {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&of, m3_fwd_kernel<float, true>, GF,
                                                        fwd_smem(4).total);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ob, m3_bwd_kernel<float, false, false>, GB,
                                                          bwd_launch_smem(chunk, 4, di.smem_per_sm));
    }
    if (e != cudaSuccess) return e;
    // the tensor-memory budget must cover every resident backward CTA
    if (ob * (int)tmem_cols_for(chunk) > 512) return cudaErrorInvalidConfiguration;
    di.occ_fwd[ai][chunk] = of > 0 ? of : 1;
    di.occ_bwd[ai][chunk] = ob > 0 ? ob : 1;
  }
  if (sms) *sms = di.sms;
  if (smem_sm) *smem_sm = di.smem_per_sm;
  if (occ_f) *occ_f = di.occ_fwd[ai][chunk];
  if (occ_b) *occ_b = di.occ_bwd[ai][chunk];
  return cudaSuccess;
}

struct Plan {
  int B, T, D, K, nc;
  int N;  // d_state
  int ldbc, lddbc;
  int Sf, mf, Sb, mb;
  size_t ckpt_bytes, ws_bytes;
  // workspace offsets (bytes)
  size_t f_aggh, f_aggs;
  size_t b_part, b_q, b_sd, b_dxpart, b_dchead;
  int ctile, cntiles;  // conv backward: steps per tile, tiles per sequence
  size_t c_part;
  int fwd_launches, bwd_launches;
  int fwd_tpc, bwd_tpc;  // threads per channel in the forward's and backward's main kernels
};

// Segments of whole chunks; every segment but the last spans >= 4 steps so
// that the conv's three-step reach crosses at most one segment boundary.
void fix_segments(int nc, int K, int want, int* S, int* m) {
  int m_min = (4 + K - 1) / K;
  if (want < 1) want = 1;
  int mm = (nc + want - 1) / want;
  if (mm < m_min) mm = m_min;
  if (mm < 1) mm = 1;
  int ss = (nc + mm - 1) / mm;
  if (ss < 1) ss = 1;
  if (ss > 65535) {
    ss = 65535;
    mm = (nc + ss - 1) / ss;
    ss = (nc + mm - 1) / mm;
  }
  *S = ss;
  *m = mm;
}

// Segment count: the largest split whose CTAs fit in `waves` waves of
// resident CTAs, with at least two chunks per segment (measured on GB300:
// the forward gains little beyond a wave or two, since its aggregate pass
// repeats most of its work; the backward keeps gaining up to several waves).
int choose_segments(int nc, int K, int64_t groups, int64_t cap, int waves) {
  if (groups < 1) groups = 1;
  int64_t want = waves * cap / groups;
  if (want < 1) want = 1;
  const int64_t max_s = (nc + 1) / 2;  // >= 2 chunks per segment
  if (want > max_s) want = max_s;
  if (want < 1) want = 1;
  int S = 1, m = 1;
  fix_segments(nc, K, (int)want, &S, &m);
  return S;
}

m3_status validate_dims(const m3_dims* dm, m3_dtype act) {
  if (!dm) return M3_ERR_NULL;
  if (act != M3_F32 && act != M3_BF16) return M3_ERR_UNSUPPORTED;
  if (dm->batch < 0 || dm->seq_len < 0 || dm->d_inner < 0 || dm->chunk < 0 || dm->segments < 0)
    return M3_ERR_DIMS;
  if ((dm->d_state != 16 && dm->d_state != 32 && dm->d_state != 64) || dm->d_conv != WC)
    return M3_ERR_UNSUPPORTED;
  // only the split kernels carry more than 16 lanes per channel
  if (dm->d_state != NS && dm->threads_per_channel == 1) return M3_ERR_UNSUPPORTED;
  if (dm->d_inner % 8 != 0) return M3_ERR_UNSUPPORTED;
  if (dm->chunk > KMAX) return M3_ERR_DIMS;
  if (dm->chunk > kmax_for(act == M3_BF16 ? 2 : 4)) return M3_ERR_UNSUPPORTED;
  if (dm->batch > 65535 || dm->seq_len > (int64_t)1 << 30 || dm->d_inner > (int64_t)1 << 24)
    return M3_ERR_DIMS;
  if (dm->segments > 65535) return M3_ERR_DIMS;
  if (dm->batch * dm->d_inner > ((int64_t)1 << 27)) return M3_ERR_DIMS;  // 1-D grid of the tail kernel
  // row strides of Bm/Cm (16-byte copies: a multiple of 16 bytes) and dB/dC
  if (dm->bc_stride < 0 || dm->dbc_stride < 0 || dm->bc_stride > ((int64_t)1 << 20) ||
      dm->dbc_stride > ((int64_t)1 << 20))
    return M3_ERR_DIMS;
  if (dm->bc_stride != 0 && dm->bc_stride < dm->d_state) return M3_ERR_DIMS;
  if (dm->dbc_stride != 0 && dm->dbc_stride < dm->d_state) return M3_ERR_DIMS;
  if (dm->bc_stride * (act == M3_BF16 ? 2 : 4) % 16 != 0) return M3_ERR_ALIGN;
  if (dm->threads_per_channel < 0 || dm->threads_per_channel > 2) return M3_ERR_UNSUPPORTED;
  return M3_OK;
}

m3_status make_plan(const m3_dims* dm, m3_dtype act, Plan* p) {
  m3_status st = validate_dims(dm, act);
  if (st != M3_OK) return st;
  p->B = (int)dm->batch;
  p->T = (int)dm->seq_len;
  p->D = (int)dm->d_inner;
  p->N = (int)dm->d_state;
  p->K = dm->chunk ? (int)dm->chunk : KDEF;
  p->nc = (p->T + p->K - 1) / p->K;
  p->ldbc = dm->bc_stride ? (int)dm->bc_stride : p->N;
  p->lddbc = dm->dbc_stride ? (int)dm->dbc_stride : p->N;
  const int groups_f = (p->D + GF - 1) / GF;
  const int groups_b = (p->D + GB - 1) / GB;
  int want_f = 1, want_b = 1;
  int64_t wave_b = 3 * 152;  // one-thread backward blocks resident at once
  int64_t wave_f = 5 * 152;  // one-thread forward blocks resident at once
  if (dm->segments > 0) {
    want_f = want_b = (int)dm->segments;
  } else if ((int64_t)p->B * p->T * p->D > 0) {
    int sms = 0, of = 0, ob = 0;
    if (note(device_info(p->K, act == M3_BF16 ? 1 : 0, &sms, &of, &ob)) != cudaSuccess)
      return M3_ERR_CUDA;
    want_f = choose_segments(p->nc, p->K, (int64_t)p->B * groups_f, (int64_t)sms * of, 2);
    want_b = choose_segments(p->nc, p->K, (int64_t)p->B * groups_b, (int64_t)sms * ob, 8);
    wave_b = (int64_t)sms * 3;  // three resident one-thread blocks per SM (measured; the
                                // occupancy query reports fewer)
    wave_f = (int64_t)sms * of;
  }
  if (p->nc == 0) {
    p->Sf = p->Sb = 1;
    p->mf = p->mb = 0;
  } else {
    fix_segments(p->nc, p->K, want_f, &p->Sf, &p->mf);
    fix_segments(p->nc, p->K, want_b, &p->Sb, &p->mb);
  }
  const size_t B = p->B, D = p->D;
  const size_t N = p->N;
  p->ckpt_bytes = B * p->nc * N * D * 4;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  // forward section
  off = 0;
  p->f_aggh = p->f_aggs = 0;
  if (p->Sf > 1) {
    p->f_aggh = take(B * p->Sf * N * D * 4);
    p->f_aggs = take(B * p->Sf * D * 4);
  }
  size_t fwd_total = off;
  // backward section (reuses the same bytes)
  off = 0;
  p->b_part = take(B * p->Sb * (N + 8) * D * 4);
  p->b_q = p->b_sd = p->b_dxpart = p->b_dchead = 0;
  if (p->Sb > 1) {
    p->b_q = take(B * p->Sb * N * D * 4);
    p->b_sd = take(B * p->Sb * D * 4);
    p->b_dxpart = take(B * p->Sb * 3 * D * 4);
    p->b_dchead = take(B * p->Sb * 3 * D * 4);
  }
  size_t bwd_total = off;
  // conv backward of the two-phase backward (its own call): CT-step tiles
  p->ctile = CT;
  p->cntiles = (p->T + CT - 1) / CT;
  off = 0;
  p->c_part = take(B * (size_t)p->cntiles * 5 * D * 4);
  const size_t conv_total = off;
  if (conv_total > bwd_total) bwd_total = conv_total;
  p->ws_bytes = fwd_total > bwd_total ? fwd_total : bwd_total;
  if (p->ws_bytes < 256) p->ws_bytes = 256;
  const bool empty = (size_t)p->B * p->T * p->D == 0;
  // d_state 16: the split kernels (two threads per channel) when the
  // one-thread grid fills less than one wave (three backward, five forward
  // blocks per SM on a 152-SM GPU, or the device's figures when the
  // segments were chosen for it); wider states: always the split kernels,
  // d_state / 8 threads per channel
  p->fwd_tpc = p->bwd_tpc = dm->threads_per_channel;
  if (p->fwd_tpc == 0) p->fwd_tpc = (int64_t)p->B * groups_f * p->Sf <= wave_f ? 2 : 1;
  if (p->bwd_tpc == 0) p->bwd_tpc = (int64_t)p->B * groups_b * p->Sb <= wave_b ? 2 : 1;
  if (p->N != NS) p->fwd_tpc = p->bwd_tpc = 2;
  if (p->fwd_tpc == 2) p->fwd_tpc = p->N / 8;
  if (p->bwd_tpc == 2) p->bwd_tpc = p->N / 8;
  p->fwd_launches = empty ? 0 : (p->Sf > 1 ? 2 : 1);
  p->bwd_launches = empty ? 0 : (p->Sb > 1 ? 3 : 2);
  return M3_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Launch with programmatic stream serialization when `pdl`: the kernel may
// begin while the previous kernel of the same call runs, and waits for it
// (grid_dep_wait) before reading its results.  The first kernel of a call
// is launched without it, so it starts after everything before it.
template <typename... Args, typename... Vals>
cudaError_t launch_k(void (*kern)(Args...), dim3 grid, unsigned block, size_t smem,
                     cudaStream_t st, bool pdl, Vals... vals) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, vals...);
}

template <typename T>
m3_status launch_fwd(const Plan& p, FwdArgs a, cudaStream_t st) {
  const int groups = (p.D + GF - 1) / GF;
  const size_t smem = fwd_smem(sizeof(T)).total;
  a.g = Geo{p.B, p.T, p.D, p.K, p.nc, p.Sf, p.mf, p.ldbc, p.lddbc};
  cudaError_t e = cudaSuccess;
  if (p.fwd_tpc != 1) {  // split kernels, N / 8 threads per channel
    const int ch = 128 / (p.N / 8);
    const dim3 ga((p.D + ch - 1) / ch, p.Sf - 1, p.B), gf((p.D + ch - 1) / ch, p.Sf, p.B);
    const size_t smem2 = fwd2_smem(sizeof(T), p.N).total;
    void (*agg)(FwdArgs) = p.N == 16 ? m3_fwd2_kernel<T, false, 16>
                         : p.N == 32 ? m3_fwd2_kernel<T, false, 32> : m3_fwd2_kernel<T, false, 64>;
    void (*fin)(FwdArgs) = p.N == 16 ? m3_fwd2_kernel<T, true, 16>
                         : p.N == 32 ? m3_fwd2_kernel<T, true, 32> : m3_fwd2_kernel<T, true, 64>;
    if (p.Sf > 1) e = launch_k(agg, ga, 128, smem2, st, false, a);
    if (e == cudaSuccess) e = launch_k(fin, gf, 128, smem2, st, p.Sf > 1, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
  }
  if (p.Sf > 1) e = launch_k(m3_fwd_kernel<T, false>, dim3(groups, p.Sf - 1, p.B), GF, smem, st, false, a);
  if (e == cudaSuccess)
    e = launch_k(m3_fwd_kernel<T, true>, dim3(groups, p.Sf, p.B), GF, smem, st, p.Sf > 1, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

// scan: stop at du (m3scan_bwd_scan); the conv side runs in launch_conv_bwd.
template <typename T>
m3_status launch_bwd(const Plan& p, BwdArgs a, cudaStream_t st, int smem_per_sm, bool scan) {
  const int groups = (p.D + GB - 1) / GB;
  a.g = Geo{p.B, p.T, p.D, p.K, p.nc, p.Sb, p.mb, p.ldbc, p.lddbc};
  cudaError_t e = cudaSuccess;
  if (p.Sb > 1) {
    // also clears dB and dC before the main kernel's reductions into them
    const bool split = p.bwd_tpc != 1;
    const int ch = split ? 128 / (p.N / 8) : GB;
    e = launch_k(agg_for<T>(split, p.N), dim3((p.D + ch - 1) / ch, p.Sb - 1, p.B), GB,
                 agg_smem(sizeof(T), p.N).total, st, false, a);
    if (note(e) != cudaSuccess) return M3_ERR_CUDA;
  } else {
    // only the d_state columns of each (batch, step) row belong to dB and dC
    const size_t pitch = (size_t)p.lddbc * 4, rows = (size_t)p.B * p.T;
    if (note(cudaMemset2DAsync(a.dB, pitch, 0, (size_t)p.N * 4, rows, st)) != cudaSuccess) return M3_ERR_CUDA;
    if (note(cudaMemset2DAsync(a.dC, pitch, 0, (size_t)p.N * 4, rows, st)) != cudaSuccess) return M3_ERR_CUDA;
  }
  const bool with_state = a.conv_in || a.g_h || a.g_conv || a.d_h_in || a.d_conv_in;
  if (p.bwd_tpc != 1) {
    a.tcols = tmem_cols2_for(p.K);
    const size_t smem = bwd2_launch_smem(p.K, sizeof(T), p.N, smem_per_sm);
    void (*kern)(BwdArgs) = scan ? (with_state ? bwd2_for<T, true, true>(p.N) : bwd2_for<T, false, true>(p.N))
                                 : (with_state ? bwd2_for<T, true, false>(p.N) : bwd2_for<T, false, false>(p.N));
    const int ch = 128 / (p.N / 8);
    e = launch_k(kern, dim3((p.D + ch - 1) / ch, p.Sb, p.B), 128, smem, st, p.Sb > 1, a);
  } else {
    a.tcols = tmem_cols_for(p.K);
    const size_t smem = bwd_launch_smem(p.K, sizeof(T), smem_per_sm);
    void (*kern)(BwdArgs) = scan ? (with_state ? m3_bwd_kernel<T, true, true> : m3_bwd_kernel<T, false, true>)
                                 : (with_state ? m3_bwd_kernel<T, true, false> : m3_bwd_kernel<T, false, false>);
    e = launch_k(kern, dim3(groups, p.Sb, p.B), GB, smem, st, p.Sb > 1, a);
  }
  // parameter outputs: N d_a_log, dD, d_dt_bias (+ d_conv_b, 4 d_conv_w)
  const int nout = scan ? p.N + 2 : p.N + 7;
  const size_t nfin = ((size_t)nout * p.D + 31) / 32;                 // 32 outputs per block
  const size_t nfix = (!scan && p.Sb > 1) ? ((size_t)p.B * (p.Sb - 1) * 3 * p.D + 255) / 256 : 0;
  if (e == cudaSuccess)
    e = launch_k(m3_bwd_tail_kernel<T>, dim3((unsigned)(nfin + nfix)), 256, 0, st, true, a,
                 p.B * p.Sb, (int)nfin, nout, p.N);
  if (e == cudaSuccess) e = cudaGetLastError();
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

// The device must have this library's kernels registered: fail early and
// cleanly when the attribute setup cannot run (no device, wrong arch).
m3_status ensure_device(int chunk, int ai, int* smem_sm) {
  int of = 0, ob = 0;
  if (note(device_info(chunk, ai, nullptr, &of, &ob, smem_sm)) != cudaSuccess) return M3_ERR_CUDA;
  return M3_OK;
}

}  // namespace

extern "C" {

const char* m3scan_status_string(m3_status s) {
  switch (s) {
    case M3_OK: return "M3_OK";
    case M3_ERR_NULL: return "M3_ERR_NULL: a required pointer is NULL";
    case M3_ERR_DIMS: return "M3_ERR_DIMS: a size is negative or out of range";
    case M3_ERR_UNSUPPORTED:
      return "M3_ERR_UNSUPPORTED: needs d_state 16, 32 or 64, d_conv 4, d_inner % 8 == 0, dtype f32 or bf16";
    case M3_ERR_ALIGN: return "M3_ERR_ALIGN: a pointer is not aligned as required";
    case M3_ERR_WORKSPACE: return "M3_ERR_WORKSPACE: workspace missing or too small";
    case M3_ERR_CUDA: return "M3_ERR_CUDA: a CUDA call or kernel launch failed";
  }
  return "unknown m3_status";
}

int32_t m3scan_version(void) { return 100; }

const char* m3scan_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda); }

m3_status m3scan_plan(const m3_dims* dims, m3_dtype act, m3_plan* out) {
  if (!out) return M3_ERR_NULL;
  Plan p;
  m3_status st = make_plan(dims, act, &p);
  if (st != M3_OK) return st;
  out->chunk = p.K;
  out->n_chunks = p.nc;
  out->fwd_segments = p.Sf;
  out->bwd_segments = p.Sb;
  out->ckpt_bytes = (int64_t)p.ckpt_bytes;
  out->workspace_bytes = (int64_t)p.ws_bytes;
  out->fwd_launches = p.fwd_launches;
  out->bwd_launches = p.bwd_launches;
  out->fwd_threads_per_channel = p.fwd_tpc;
  out->bwd_threads_per_channel = p.bwd_tpc;
  return M3_OK;
}

}  // extern "C"

namespace {

// A window with no steps: the state outputs are the state inputs (zero when
// absent), and the state-input gradients are the upstream gradients.
m3_status pass_state(const void* in, void* out, size_t bytes, cudaStream_t s) {
  if (!out || bytes == 0) return M3_OK;
  const cudaError_t e = in ? cudaMemcpyAsync(out, in, bytes, cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(out, 0, bytes, s);
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

// Alignment of the carried-state pointers: f32 arrays 4 bytes, activation
// arrays one element.
bool state_aligned(const void* f32a, const void* f32b, const void* acta, const void* actb,
                   m3_dtype act) {
  const size_t ea = act == M3_BF16 ? 2 : 4;
  return aligned(f32a, 4) && aligned(f32b, 4) && aligned(acta, ea) && aligned(actb, ea);
}

m3_status fwd_impl(const m3_dims* dims, m3_dtype act, const void* x, const void* delta_raw,
                   const void* z, const void* Bm, const void* Cm, const float* conv_w,
                   const float* conv_b, const float* dt_bias, const float* a_log, const float* D,
                   void* gated, void* y_dbg, float* ckpt, const m3_fwd_state* state,
                   void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  Plan p;
  m3_status st = make_plan(dims, act, &p);
  if (st != M3_OK) return st;
  const m3_fwd_state none{};
  const m3_fwd_state& sv = state ? *state : none;
  if (!state_aligned(sv.ssm_state, sv.ssm_state_out, sv.conv_state, sv.conv_state_out, act))
    return M3_ERR_ALIGN;
  if ((size_t)p.B * p.T * p.D == 0) {
    const size_t bd = (size_t)p.B * p.D;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = pass_state(sv.ssm_state, sv.ssm_state_out, bd * p.N * 4, s);
    if (st == M3_OK) st = pass_state(sv.conv_state, sv.conv_state_out, bd * 3 * (act == M3_BF16 ? 2 : 4), s);
    return st;
  }
  if (!x || !delta_raw || !z || !Bm || !Cm || !conv_w || !conv_b || !dt_bias || !a_log || !D ||
      !gated || !ckpt)
    return M3_ERR_NULL;
  const void* act_ptrs[] = {x, delta_raw, z, Bm, Cm, gated, y_dbg};
  for (const void* q : act_ptrs)
    if (q && !aligned(q, 16)) return M3_ERR_ALIGN;
  const void* f_ptrs[] = {conv_w, conv_b, dt_bias, a_log, D};
  for (const void* q : f_ptrs)
    if (!aligned(q, 4)) return M3_ERR_ALIGN;
  if (!aligned(ckpt, 16)) return M3_ERR_ALIGN;
  if (p.Sf > 1) {
    if (!workspace) return M3_ERR_WORKSPACE;
    if (workspace_bytes < p.ws_bytes) return M3_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return M3_ERR_ALIGN;
  }
  int smem_sm = 0;
  if (ensure_device(p.K, act == M3_BF16 ? 1 : 0, &smem_sm) != M3_OK) return M3_ERR_CUDA;
  FwdArgs a{};
  a.x = x; a.dr = delta_raw; a.z = z; a.Bm = Bm; a.Cm = Cm;
  a.conv_w = conv_w; a.conv_b = conv_b; a.dt_bias = dt_bias; a.a_log = a_log; a.Dp = D;
  a.gated = gated; a.y_dbg = y_dbg; a.ckpt = ckpt;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.agg_h = p.Sf > 1 ? reinterpret_cast<float*>(ws + p.f_aggh) : nullptr;
  a.agg_s = p.Sf > 1 ? reinterpret_cast<float*>(ws + p.f_aggs) : nullptr;
  a.h_in = sv.ssm_state; a.conv_in = sv.conv_state;
  a.h_out = sv.ssm_state_out; a.conv_out = sv.conv_state_out;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return act == M3_BF16 ? launch_fwd<__nv_bfloat16>(p, a, s) : launch_fwd<float>(p, a, s);
}

m3_status bwd_impl(const m3_dims* dims, m3_dtype act, const void* x, const void* delta_raw,
                   const void* z, const void* Bm, const void* Cm, const float* conv_w,
                   const float* conv_b, const float* dt_bias, const float* a_log, const float* D,
                   const float* ckpt, const void* d_gated, void* d_x, void* d_delta_raw, void* dz,
                   void* du_dbg, float* dB, float* dC, float* d_conv_w, float* d_conv_b,
                   float* d_dt_bias, float* d_a_log, float* dD, const m3_bwd_state* state,
                   void* workspace, size_t workspace_bytes, m3_stream_t stream, bool scan) {
  Plan p;
  m3_status st = make_plan(dims, act, &p);
  if (st != M3_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const m3_bwd_state none{};
  const m3_bwd_state& sv = state ? *state : none;
  if (!state_aligned(sv.d_ssm_state_out, sv.d_ssm_state, sv.conv_state, sv.d_conv_state_out, act) ||
      !aligned(sv.d_conv_state, act == M3_BF16 ? 2 : 4))
    return M3_ERR_ALIGN;
  if ((size_t)p.B * p.T * p.D == 0) {
    const size_t bd = (size_t)p.B * p.D;
    st = pass_state(sv.d_ssm_state_out, sv.d_ssm_state, bd * p.N * 4, s);
    if (st == M3_OK)
      st = pass_state(sv.d_conv_state_out, sv.d_conv_state, bd * 3 * (act == M3_BF16 ? 2 : 4), s);
    if (st != M3_OK) return st;
    // no elements: parameter grads are zero (or unchanged when accumulating)
    if (p.D > 0 && !dims->accumulate_param_grads) {
      if ((!scan && (!d_conv_w || !d_conv_b)) || !d_dt_bias || !d_a_log || !dD) return M3_ERR_NULL;
      const size_t D_ = p.D;
      if ((!scan && (cudaMemsetAsync(d_conv_w, 0, D_ * WC * 4, s) != cudaSuccess ||
                     cudaMemsetAsync(d_conv_b, 0, D_ * 4, s) != cudaSuccess)) ||
          cudaMemsetAsync(d_dt_bias, 0, D_ * 4, s) != cudaSuccess ||
          cudaMemsetAsync(d_a_log, 0, D_ * p.N * 4, s) != cudaSuccess ||
          cudaMemsetAsync(dD, 0, D_ * 4, s) != cudaSuccess) {
        note(cudaGetLastError());
        return M3_ERR_CUDA;
      }
    }
    return M3_OK;
  }
  if (!x || !delta_raw || !z || !Bm || !Cm || !conv_w || !conv_b || !dt_bias || !a_log || !D ||
      !ckpt || !d_gated || !d_delta_raw || !dz || !dB || !dC || !d_dt_bias || !d_a_log || !dD)
    return M3_ERR_NULL;
  if (scan ? !du_dbg : (!d_x || !d_conv_w || !d_conv_b)) return M3_ERR_NULL;
  const void* act_ptrs[] = {x, delta_raw, z, Bm, Cm, d_gated, d_x, d_delta_raw, dz, du_dbg};
  for (const void* q : act_ptrs)
    if (q && !aligned(q, 16)) return M3_ERR_ALIGN;
  const void* f_ptrs[] = {conv_w, conv_b, dt_bias, a_log, D, dB, dC,
                          d_conv_w, d_conv_b, d_dt_bias, d_a_log, dD};
  for (const void* q : f_ptrs)
    if (!aligned(q, 4)) return M3_ERR_ALIGN;
  if (!aligned(ckpt, 16)) return M3_ERR_ALIGN;
  if (!workspace) return M3_ERR_WORKSPACE;
  if (workspace_bytes < p.ws_bytes) return M3_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return M3_ERR_ALIGN;
  int smem_sm = 0;
  if (ensure_device(p.K, act == M3_BF16 ? 1 : 0, &smem_sm) != M3_OK) return M3_ERR_CUDA;
  BwdArgs a{};
  a.x = x; a.dr = delta_raw; a.z = z; a.Bm = Bm; a.Cm = Cm; a.dg = d_gated;
  a.conv_w = conv_w; a.conv_b = conv_b; a.dt_bias = dt_bias; a.a_log = a_log; a.Dp = D;
  a.ckpt = ckpt;
  a.dx = d_x; a.ddr = d_delta_raw; a.dz = dz; a.du_dbg = du_dbg;
  a.dB = dB; a.dC = dC;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.partials = reinterpret_cast<float*>(ws + p.b_part);
  if (p.Sb > 1) {
    a.q = reinterpret_cast<float*>(ws + p.b_q);
    a.sd = reinterpret_cast<float*>(ws + p.b_sd);
    a.dxpart = reinterpret_cast<float*>(ws + p.b_dxpart);
    a.dchead = reinterpret_cast<float*>(ws + p.b_dchead);
  }
  a.d_conv_w = d_conv_w; a.d_conv_b = d_conv_b; a.d_dt_bias = d_dt_bias; a.d_a_log = d_a_log;
  a.dD = dD;
  a.accumulate = dims->accumulate_param_grads ? 1 : 0;
  a.conv_in = sv.conv_state; a.g_h = sv.d_ssm_state_out; a.g_conv = sv.d_conv_state_out;
  a.d_h_in = sv.d_ssm_state; a.d_conv_in = sv.d_conv_state;
  m3_status r = act == M3_BF16 ? launch_bwd<__nv_bfloat16>(p, a, s, smem_sm, scan)
                                : launch_bwd<float>(p, a, s, smem_sm, scan);
  if (r != M3_OK) cudaGetLastError();
  return r;
}

}  // namespace

extern "C" {

m3_status m3scan_fwd(const m3_dims* dims, m3_dtype act, const void* x, const void* delta_raw,
                     const void* z, const void* Bm, const void* Cm, const float* conv_w,
                     const float* conv_b, const float* dt_bias, const float* a_log, const float* D,
                     void* gated, void* y_dbg, float* ckpt, void* workspace, size_t workspace_bytes,
                     m3_stream_t stream) {
  return fwd_impl(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, gated,
                  y_dbg, ckpt, nullptr, workspace, workspace_bytes, stream);
}

m3_status m3scan_fwd_state(const m3_dims* dims, m3_dtype act, const void* x,
                           const void* delta_raw, const void* z, const void* Bm, const void* Cm,
                           const float* conv_w, const float* conv_b, const float* dt_bias,
                           const float* a_log, const float* D, void* gated, void* y_dbg,
                           float* ckpt, const m3_fwd_state* state, void* workspace,
                           size_t workspace_bytes, m3_stream_t stream) {
  if (!state) return M3_ERR_NULL;
  return fwd_impl(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, gated,
                  y_dbg, ckpt, state, workspace, workspace_bytes, stream);
}

m3_status m3scan_bwd(const m3_dims* dims, m3_dtype act, const void* x, const void* delta_raw,
                     const void* z, const void* Bm, const void* Cm, const float* conv_w,
                     const float* conv_b, const float* dt_bias, const float* a_log, const float* D,
                     const float* ckpt, const void* d_gated, void* d_x, void* d_delta_raw, void* dz,
                     void* du_dbg, float* dB, float* dC, float* d_conv_w, float* d_conv_b,
                     float* d_dt_bias, float* d_a_log, float* dD, void* workspace,
                     size_t workspace_bytes, m3_stream_t stream) {
  return bwd_impl(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                  d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b, d_dt_bias,
                  d_a_log, dD, nullptr, workspace, workspace_bytes, stream, false);
}

m3_status m3scan_bwd_state(const m3_dims* dims, m3_dtype act, const void* x,
                           const void* delta_raw, const void* z, const void* Bm, const void* Cm,
                           const float* conv_w, const float* conv_b, const float* dt_bias,
                           const float* a_log, const float* D, const float* ckpt,
                           const void* d_gated, void* d_x, void* d_delta_raw, void* dz,
                           void* du_dbg, float* dB, float* dC, float* d_conv_w, float* d_conv_b,
                           float* d_dt_bias, float* d_a_log, float* dD,
                           const m3_bwd_state* state, void* workspace, size_t workspace_bytes,
                           m3_stream_t stream) {
  if (!state) return M3_ERR_NULL;
  return bwd_impl(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                  d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b, d_dt_bias,
                  d_a_log, dD, state, workspace, workspace_bytes, stream, false);
}

m3_status m3scan_bwd_scan(const m3_dims* dims, m3_dtype act, const void* x, const void* delta_raw,
                          const void* z, const void* Bm, const void* Cm, const float* conv_w,
                          const float* conv_b, const float* dt_bias, const float* a_log,
                          const float* D, const float* ckpt, const void* d_gated, void* du,
                          void* d_delta_raw, void* dz, float* dB, float* dC, float* d_dt_bias,
                          float* d_a_log, float* dD, const m3_bwd_state* state, void* workspace,
                          size_t workspace_bytes, m3_stream_t stream) {
  return bwd_impl(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                  d_gated, nullptr, d_delta_raw, dz, du, dB, dC, nullptr, nullptr, d_dt_bias,
                  d_a_log, dD, state, workspace, workspace_bytes, stream, true);
}

m3_status m3scan_conv_bwd(const m3_dims* dims, m3_dtype act, const void* x, const float* conv_w,
                          const float* conv_b, const void* du, const void* du_extra, void* d_x,
                          float* d_conv_w, float* d_conv_b, const m3_bwd_state* state,
                          void* workspace, size_t workspace_bytes, m3_stream_t stream) {
  Plan p;
  m3_status st = make_plan(dims, act, &p);
  if (st != M3_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const m3_bwd_state none{};
  const m3_bwd_state& sv = state ? *state : none;
  const size_t es = act == M3_BF16 ? 2 : 4;
  if (!aligned(sv.conv_state, es) || !aligned(sv.d_conv_state_out, es) || !aligned(sv.d_conv_state, es))
    return M3_ERR_ALIGN;
  if ((size_t)p.B * p.T * p.D == 0) {
    st = pass_state(sv.d_conv_state_out, sv.d_conv_state, (size_t)p.B * p.D * 3 * es, s);
    if (st != M3_OK) return st;
    if (p.D > 0 && !dims->accumulate_param_grads) {
      if (!d_conv_w || !d_conv_b) return M3_ERR_NULL;
      if (note(cudaMemsetAsync(d_conv_w, 0, (size_t)p.D * WC * 4, s)) != cudaSuccess ||
          note(cudaMemsetAsync(d_conv_b, 0, (size_t)p.D * 4, s)) != cudaSuccess)
        return M3_ERR_CUDA;
    }
    return M3_OK;
  }
  if (!x || !conv_w || !conv_b || !du || !d_x || !d_conv_w || !d_conv_b) return M3_ERR_NULL;
  const void* act_ptrs[] = {x, du, du_extra, d_x};
  for (const void* q : act_ptrs)
    if (q && !aligned(q, 16)) return M3_ERR_ALIGN;
  const void* f_ptrs[] = {conv_w, conv_b, d_conv_w, d_conv_b};
  for (const void* q : f_ptrs)
    if (!aligned(q, 4)) return M3_ERR_ALIGN;
  if (!workspace || workspace_bytes < p.ws_bytes) return M3_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return M3_ERR_ALIGN;
  int smem_sm = 0;
  if (ensure_device(p.K, act == M3_BF16 ? 1 : 0, &smem_sm) != M3_OK) return M3_ERR_CUDA;
  ConvArgs a{};
  a.B = p.B; a.T = p.T; a.D = p.D; a.tile = p.ctile; a.ntiles = p.cntiles;
  a.x = x; a.du = du; a.du_extra = du_extra; a.conv_w = conv_w; a.conv_b = conv_b; a.dx = d_x;
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + p.c_part);
  a.conv_in = sv.conv_state; a.g_conv = sv.d_conv_state_out; a.d_conv_in = sv.d_conv_state;
  a.d_conv_w = d_conv_w; a.d_conv_b = d_conv_b;
  a.accumulate = dims->accumulate_param_grads ? 1 : 0;
  const dim3 grid((unsigned)((p.D + 127) / 128), (unsigned)p.cntiles, (unsigned)p.B);
  cudaError_t e = act == M3_BF16
                      ? launch_k(m3_conv_bwd_kernel<__nv_bfloat16>, grid, 128, conv_smem(2).total, s, false, a)
                      : launch_k(m3_conv_bwd_kernel<float>, grid, 128, conv_smem(4).total, s, false, a);
  if (e == cudaSuccess)
    e = launch_k(m3_conv_fin_kernel, dim3((unsigned)((5 * (size_t)p.D + 31) / 32)), 256, 0, s, true, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}


}  // extern "C"

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64];  // device address of g_noalloc_scratch, per device

// Set-up for m3scan_bwd_noalloc, once per device with that device current:
// look up the device address of the library's scratch array.
m3_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return M3_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      note(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return M3_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return M3_OK;
}

}  // namespace

extern "C" {

// The backward of m3scan_bwd, run on the library's own fixed scratch array
// instead of a caller-provided workspace; it allocates nothing.  Nothing in
// the scratch has to start at zero: every byte the kernels read in one call
// is written earlier in the same call.
m3_status m3scan_bwd_noalloc(const m3_dims* dims, m3_dtype act, const void* x,
                             const void* delta_raw, const void* z, const void* Bm,
                             const void* Cm, const float* conv_w, const float* conv_b,
                             const float* dt_bias, const float* a_log, const float* D,
                             const float* ckpt, const void* d_gated, void* d_x,
                             void* d_delta_raw, void* dz, void* du_dbg, float* dB, float* dC,
                             float* d_conv_w, float* d_conv_b, float* d_dt_bias,
                             float* d_a_log, float* dD, m3_stream_t stream) {
  Plan p;
  m3_status st = make_plan(dims, act, &p);
  if (st != M3_OK) return st;
  if (p.ws_bytes > (size_t)M3SCAN_NOALLOC_SCRATCH_BYTES) return M3_ERR_WORKSPACE;
  void* ws = nullptr;
  if ((size_t)p.B * p.T * p.D > 0) {
    st = noalloc_scratch(&ws);
    if (st != M3_OK) return st;
  }
  return m3scan_bwd(dims, act, x, delta_raw, z, Bm, Cm, conv_w, conv_b, dt_bias, a_log, D, ckpt,
                    d_gated, d_x, d_delta_raw, dz, du_dbg, dB, dC, d_conv_w, d_conv_b, d_dt_bias,
                    d_a_log, dD, ws, (size_t)M3SCAN_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"

namespace {

template <typename T, int N, int R>
cudaError_t launch_decode_r(const DecArgs& a, cudaStream_t st) {
  constexpr int CH = GD / (N / 16);
  m3_decode_kernel<T, N, R>
      <<<dim3((unsigned)((a.D + CH - 1) / CH), (unsigned)((a.B + R - 1) / R)), GD, 0, st>>>(a);
  return cudaGetLastError();
}

// Two batch rows per thread when there are still enough blocks to give
// every SM several (a small batch keeps one row per thread, for more blocks).
template <typename T, int N>
cudaError_t launch_decode(const DecArgs& a, cudaStream_t st, int sms) {
  constexpr int CH = GD / (N / 16);
  const int64_t blocks2 = (int64_t)((a.D + CH - 1) / CH) * ((a.B + 1) / 2);
  if (blocks2 >= 4 * (int64_t)sms) return launch_decode_r<T, N, 2>(a, st);
  return launch_decode_r<T, N, 1>(a, st);
}

template <typename T>
cudaError_t launch_decode_n(int n, const DecArgs& a, cudaStream_t st, int sms) {
  if (n == 16) return launch_decode<T, 16>(a, st, sms);
  if (n == 32) return launch_decode<T, 32>(a, st, sms);
  return launch_decode<T, 64>(a, st, sms);
}

}  // namespace

extern "C" {

// The forward of a short window from the carried state, updating the state
// in place (no checkpoints, no workspace).
m3_status m3scan_decode(const m3_dims* dims, m3_dtype act, const void* x, const void* delta_raw,
                        const void* z, const void* Bm, const void* Cm, const float* conv_w,
                        const float* conv_b, const float* dt_bias, const float* a_log,
                        const float* D, float* ssm_state, void* conv_state, void* gated,
                        void* y_dbg, m3_stream_t stream) {
  if (!dims) return M3_ERR_NULL;
  if (act != M3_F32 && act != M3_BF16) return M3_ERR_UNSUPPORTED;
  if (dims->batch < 0 || dims->seq_len < 0 || dims->d_inner < 0) return M3_ERR_DIMS;
  if ((dims->d_state != 16 && dims->d_state != 32 && dims->d_state != 64) || dims->d_conv != WC)
    return M3_ERR_UNSUPPORTED;
  if (dims->batch > 65535 || dims->seq_len > ((int64_t)1 << 30) || dims->d_inner > ((int64_t)1 << 24))
    return M3_ERR_DIMS;
  if (dims->bc_stride < 0 || dims->bc_stride > ((int64_t)1 << 20) ||
      (dims->bc_stride != 0 && dims->bc_stride < dims->d_state))
    return M3_ERR_DIMS;
  if (dims->batch * dims->seq_len * dims->d_inner == 0) return M3_OK;
  if (!x || !delta_raw || !z || !Bm || !Cm || !conv_w || !conv_b || !dt_bias || !a_log || !D ||
      !ssm_state || !conv_state || !gated)
    return M3_ERR_NULL;
  const size_t es = act == M3_BF16 ? 2 : 4;
  const void* act_ptrs[] = {x, delta_raw, z, Bm, Cm, conv_state, gated, y_dbg};
  for (const void* q : act_ptrs)
    if (!aligned(q, es)) return M3_ERR_ALIGN;
  const void* f_ptrs[] = {conv_w, conv_b, dt_bias, a_log, D, ssm_state};
  for (const void* q : f_ptrs)
    if (!aligned(q, 4)) return M3_ERR_ALIGN;
  DecArgs a{};
  a.B = (int)dims->batch;
  a.T = (int)dims->seq_len;
  a.D = (int)dims->d_inner;
  a.ldbc = dims->bc_stride ? (int)dims->bc_stride : (int)dims->d_state;
  a.x = x; a.dr = delta_raw; a.z = z; a.Bm = Bm; a.Cm = Cm;
  a.conv_w = conv_w; a.conv_b = conv_b; a.dt_bias = dt_bias; a.a_log = a_log; a.Dp = D;
  a.h = ssm_state; a.conv = conv_state; a.gated = gated; a.y_dbg = y_dbg;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int n = (int)dims->d_state;
  int sms = 0, of = 0, ob = 0;
  if (note(device_info(KDEF, act == M3_BF16 ? 1 : 0, &sms, &of, &ob)) != cudaSuccess)
    return M3_ERR_CUDA;
  const cudaError_t e = act == M3_BF16 ? launch_decode_n<__nv_bfloat16>(n, a, s, sms)
                                       : launch_decode_n<float>(n, a, s, sms);
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

}  // extern "C"

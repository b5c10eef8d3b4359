// m3_common.cuh -- selective-scan layer core (Mamba-1) for sm_103a.
// Shared by the library's translation units: constants, device helpers,
// kernel argument structs, shared-memory layouts, the launch plan and the
// entry points each unit provides to the others.
#pragma once

#include <cuda.h>  // CUtensorMap (the driver function that fills one is looked up at run time)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/m3scan.h"

namespace m3 {

constexpr int NS = 16;        // d_state lanes per channel
constexpr int WC = 4;         // conv taps
constexpr int GF = 128;       // forward: channels (= threads) per block
constexpr int GB = 128;       // backward: channels (= threads) per block = 4 warps,
                              // one per tensor-memory lane quadrant
constexpr int NWB = GB / 32;  // backward warps per block
constexpr int TT = 8;         // one-thread forward / aggregate staging tile (steps):
                              // the small footprint lets more blocks stay resident
constexpr int TT2 = 16;       // the split kernels' staging tile: they serve grids under
                              // a wave, where fewer, longer tiles wait less
constexpr int SUB = 8;        // forward scalar sub-tile (steps)
constexpr int KT = 8;         // backward tile: steps whose states are recomputed on chip at once
constexpr int KMAX = 256;     // largest checkpoint interval
constexpr int KLONG = 64;     // default checkpoint interval of long sequences
constexpr int KSHORT = 8;     // default checkpoint interval of short sequences
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

// softplus(v) (.x) and sigmoid(v) (.y) from one exponential e = e^-|v|:
// softplus as in softplus_f below; sigmoid(v) = 1 / (1 + e) for v >= 0 and
// e / (1 + e) for v < 0.
__device__ __forceinline__ float2 softplus_sigmoid(float v) {
  const float e = ex2(-fabsf(v) * LOG2E);
  const float series = e * fmaf(e, fmaf(e, 0.33333334f, -0.5f), 1.0f);
  const float lg = lg2_a(1.0f + e) * LN2;
  const float r = rcp_a(1.0f + e);
  return make_float2(fmaxf(v, 0.0f) + (e < 0.015625f ? series : lg), v >= 0.0f ? r : e * r);
}

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
// The same load and store split from their waits, with no memory clobber:
// ordinary loads and stores may be scheduled across them.  The wait names
// the loaded registers as read-written, so no use of them can move above it.
__device__ __forceinline__ void tmem_st16_async(uint32_t taddr, const float2 (&v)[NS / 2]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y),
      "f"(v[3].x), "f"(v[3].y), "f"(v[4].x), "f"(v[4].y), "f"(v[5].x), "f"(v[5].y), "f"(v[6].x),
      "f"(v[6].y), "f"(v[7].x), "f"(v[7].y));
}
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, float2 (&v)[NS / 2]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=f"(v[0].x), "=f"(v[0].y), "=f"(v[1].x), "=f"(v[1].y), "=f"(v[2].x), "=f"(v[2].y),
        "=f"(v[3].x), "=f"(v[3].y), "=f"(v[4].x), "=f"(v[4].y), "=f"(v[5].x), "=f"(v[5].y),
        "=f"(v[6].x), "=f"(v[6].y), "=f"(v[7].x), "=f"(v[7].y) : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(float2 (&v)[NS / 2]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0].x), "+f"(v[0].y), "+f"(v[1].x), "+f"(v[1].y), "+f"(v[2].x), "+f"(v[2].y),
                 "+f"(v[3].x), "+f"(v[3].y), "+f"(v[4].x), "+f"(v[4].y), "+f"(v[5].x), "+f"(v[5].y),
                 "+f"(v[6].x), "+f"(v[6].y), "+f"(v[7].x), "+f"(v[7].y));
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

// ---- tile copies by the tensor memory accelerator ----
// One thread issues cp.async.bulk.tensor copies of whole tiles into shared
// memory; they complete on a shared-memory mbarrier whose transaction count
// the issuing thread raised by the tiles' bytes.  Elements outside the
// tensor (negative or too-large coordinates) arrive as zeros.
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// makes initialised mbarriers visible to the copy engine (before a block barrier)
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait until the phase of the given parity has completed.  Gives up and
// returns false after about one second, so a copy that never lands cannot
// hang the GPU; the caller then reports the failure and leaves.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(a), "r"(parity) : "memory");
    if (done) return true;
    if (i == 0) t0 = global_ns();
    else if (global_ns() - t0 > 1000000000ull) return false;
  }
}
// A kernel that gave up waiting for a tile copy records it in its
// translation unit's per-device word and, when the call has a workspace, in
// that workspace's status block (bits are only ever set on the device; the
// host reads and clears them).
__device__ __forceinline__ void report_timeout(unsigned* unit_word, unsigned* ws_word) {
  atomicOr(unit_word, 1u);
  if (ws_word) atomicOr(ws_word, 1u);
}

// orders this thread's view of earlier generic-proxy shared-memory accesses
// (made visible to it by a block barrier) before its next tile copies
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
// Tile store from shared memory (elements outside the tensor are not
// written); the issuing thread commits a bulk group after its stores.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared memory read by every committed bulk store may be overwritten
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk store has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// orders this thread's generic-proxy writes to global memory before later
// tile copies (async proxy) that read them
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// A 64-bit L2 cache policy that keeps written lines resident in preference
// to others (for short-lived workspace data read back soon), and stores
// that carry it.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
      : "memory");
}

// Thread-block cluster: a barrier over every thread of every block in the
// cluster (the release / acquire halves order shared and global memory
// writes before it against reads after it), and loads from another block's
// shared memory at the same offset.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The same without the release half: for a barrier whose only job is that
// no block leaves before the others have used the values they loaded from
// its shared memory (a load whose value was consumed has completed).
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

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

// Chain segment aggregates into v (NP lane pairs): for cnt segments
// sp = first, first + step, ...:  v = exp2(sum_delta(sp) a2) v + local(sp),
// with sum_delta at sums[(bS + sp) D + d] and the local lane pair P at
// locs[((bS + sp) N + lane(P)) D + d] (and the next row).  The loads of CB
// segments are issued before their multiply-adds, so a chain of cnt
// segments waits for about cnt / CB memory round trips, not cnt.
template <int NP, int CB, typename Lane>
__device__ __forceinline__ void chain_segments(float2 (&v)[NP], const float2 (&a2)[NP],
                                               const float* __restrict__ sums,
                                               const float* __restrict__ locs, int N, size_t bS,
                                               int first, int step, int cnt, int D, int d,
                                               bool active, Lane lane) {
  for (int i0 = 0; i0 < cnt; i0 += CB) {
    float dl[CB];
    float2 loc[CB][NP];
#pragma unroll
    for (int k = 0; k < CB; ++k) {
      const bool ok = active && i0 + k < cnt;
      const size_t bs = bS + (ok ? first + (i0 + k) * step : 0);
      dl[k] = ok ? sums[bs * D + d] : 0.f;
#pragma unroll
      for (int P = 0; P < NP; ++P) {
        const float* l = locs + (bs * N + lane(P)) * D + d;
        loc[k][P] = ok ? make_float2(l[0], l[D]) : make_float2(0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < CB; ++k) {
      if (i0 + k < cnt) {
        const float2 dl2 = f2b(dl[k]);
#pragma unroll
        for (int P = 0; P < NP; ++P) v[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), v[P], loc[k][P]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// geometry and kernel arguments
// ---------------------------------------------------------------------------

struct Geo {
  int B, T, D, K, nc, S, m;  // S segments of m chunks (the last may be short)
  int ldbc, lddbc;           // row strides (elements) of Bm/Cm and of dB/dC
  // backward: tiles of KS = min(K, KT) steps; nsk = sub-checkpoints per chunk
  // kept in the workspace (the states before tiles 1 .. ceil(K / KS) - 2)
  int KS, nsk;
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
  // the workspace's status block (nullable: no workspace)
  unsigned* status;
  // tile maps of the forward's staging and stores (see TF_* below)
  CUtensorMap tm[7];
};
// tensor maps of FwdArgs::tm: activations [B, T, D] with boxes of the
// block's channels x TT rows (TT2 in the split kernels, whose x boxes add
// the three conv halo rows); B and C [B, T, ld] with boxes of N x TT (TT2); stores of
// the one-thread final pass: gated and y [B, T, D] with boxes of GF x SUB
enum { TF_X = 0, TF_DR, TF_Z, TF_B, TF_C, TF_OG, TF_OY };

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
  // deterministic dB/dC: per-(batch, step, channel block) partials
  // [B * T][nblk][2N], summed by m3_dbc_sum_kernel; NULL: float atomics
  float* dbc_part;
  int nblk;
  // 1: the split main kernel runs with the S segments of a (channel block,
  // batch) as one thread-block cluster, which sums its parameter shares over
  // the segments and adds them into the outputs (cleared by the aggregate
  // kernel unless accumulating) and finishes d_x at the segment boundaries
  int fin;
  // the workspace's status block
  unsigned* status;
  // sub-checkpoints of the chunk a block is working on, [blocks][nsk][N][ch]
  // f32 (block = linear block index; ch = channels per block)
  float* sk;
  // tile maps of the backward's staging and stores (see TM_* below)
  CUtensorMap tm[16];
};
// The backward's last kernel needs only these (a small argument block keeps
// its launch cheap).
struct TailArgs {
  Geo g;
  const float *partials, *dxpart, *dchead, *conv_w, *a_log;
  void* dx;
  float *d_a_log, *dD, *d_dt_bias, *d_conv_b, *d_conv_w;
  int accumulate;
};

// tensor maps of BwdArgs::tm, boxes of the block's channels (128 / threads
// per channel): main kernels -- activations [B, T, D] x (KS + 3) rows (x)
// or KS rows, B and C [B, T, ld] N x KS, checkpoints [B, nc, N, D] f32
// channels x N, sub-checkpoints [blocks, nsk, N, ch] f32 ch x N;
// aggregate kernel -- delta_raw, z, d_gated TT rows (TT2 for d_state / 8
// threads per channel), C N x TT (TT2); stores of
// the one-thread main kernel -- dz, d_delta_raw, d_x, du [B, T, D] x KS rows
enum { TM_X = 0, TM_DR, TM_Z, TM_DG, TM_B, TM_C, TM_CK, TM_ADR, TM_AZ, TM_ADG, TM_AC, TM_SK,
       TM_ODZ, TM_ODR, TM_ODX, TM_ODU };

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
// buffers {x: [TT2+3][CH] (three halo rows), delta_raw, z: [TT2][CH]; B, C:
// [TT2][N]}, float B and C of the tile, and per-step scalars sc[SUB][CH]
// float4 shared by the threads of a channel.
struct Fwd2Smem {
  size_t x, dr, z, Bt, Ct, tile, fB, fC, sc, total;
};
__host__ __device__ inline Fwd2Smem fwd2_smem(int es, int N) {
  const int CH = 128 / (N / 8);  // channels per block
  Fwd2Smem s;
  s.x = 0;
  s.dr = s.x + align_up((size_t)(TT2 + 3) * CH * es, 128);
  s.z = s.dr + align_up((size_t)TT2 * CH * es, 128);
  s.Bt = s.z + align_up((size_t)TT2 * CH * es, 128);
  s.Ct = s.Bt + align_up((size_t)TT2 * N * es, 128);
  s.tile = s.Ct + align_up((size_t)TT2 * N * es, 128);
  s.fB = 2 * s.tile;
  s.fC = s.fB + (size_t)TT2 * N * 4;
  s.sc = s.fC + (size_t)TT2 * N * 4;
  s.total = s.sc + (size_t)SUB * CH * 16;
  return s;
}

// Backward shared memory for tiles of K steps: two staging buffers {x:
// [K+3][GB] (three halo rows before the tile), delta_raw, z, d_gated: [K][GB]
// act; B, C: [K][16] act; the tile's start state ck: [16][GB] f32}; B and C
// of the current tile as float (the recomputed states live in tensor memory,
// see m3_bwd_kernel);
// per-step scalars, two thread-private float4 slots per step: s0[K][GB] =
// (delta, delta*u, dy, dz factor -> sum_n A dh exp(delta A) h_{t-1}) and
// s1[K][GB] = (D*u -> sum_n dh B, sigmoid(delta_raw + dt_bias), sigmoid(c),
// c); per-warp dB/dC sums red[K][NWB][32].
// The split backward keeps B and C of a chunk as float in NROT = 4 copies
// whose lane pairs are permuted the way the threads' state registers are
// (see m3_bwd2_kernel), so every thread reads its copy in register order at
// fixed offsets.  Copy r starts r * rot_stride(K, N) floats in: 16 bytes
// past a multiple of 128, so the copies that a warp's threads read at the
// same offset fall in different banks.
constexpr int NROT = 4;
__host__ __device__ inline int rot_stride(int K, int N) { return K * N + 4; }
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
  s.fC = s.fB + (size_t)NROT * rot_stride(K, N) * 4;
  s.scal = s.fC + (size_t)NROT * rot_stride(K, N) * 4;
  s.dcs = s.scal + (size_t)2 * K * CH * 16;
  s.red = s.dcs + align_up((size_t)(K + 3) * CH * 4, 128);
  s.total = s.red + (size_t)K * 4 * 2 * N * 4;
  return s;
}

// Backward aggregate shared memory for tiles of tt steps: two buffers
// {delta_raw, z, d_gated: [tt][GB]; C: [tt][N]}, float C and per-step
// (delta, dy) [tt][GB] float2.
struct AggSmem {
  size_t dr, z, dg, Ct, tile, fC, sc, total;
};
__host__ __device__ inline AggSmem agg_smem(int es, int N, int tt) {
  AggSmem s;
  s.dr = 0;
  s.z = s.dr + align_up((size_t)tt * GB * es, 128);
  s.dg = s.z + align_up((size_t)tt * GB * es, 128);
  s.Ct = s.dg + align_up((size_t)tt * GB * es, 128);
  s.tile = s.Ct + align_up((size_t)tt * N * es, 128);
  s.fC = 2 * s.tile;
  s.sc = s.fC + (size_t)tt * N * 4;
  s.total = s.sc + (size_t)tt * GB * 8;
  return s;
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
  unsigned* status;  // the workspace's status block
  // tile maps: x [B, T, D] with boxes of 128 channels x (CT + 6) rows, du
  // and du_extra with 128 x (CT + 3)
  CUtensorMap tm[3];
};

// Steps per conv-backward tile: rows [t0 - 3, t0 + CT + 3) of x and
// [t0, t0 + CT + 3) of du and du_extra arrive in shared memory by tensor-map
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
  // tile map of h (boxes of the block's channels x N lanes x its batch rows),
  // used when h is 16-byte aligned and d_inner a multiple of 4
  CUtensorMap tm_h;
};

constexpr int GD = 128;  // decode: channels (= threads) per block


// ---------------------------------------------------------------------------
// host side: sizes, the plan, launching
// ---------------------------------------------------------------------------

// the workspace's status block (M3SCAN_STATUS_BYTES) comes first
constexpr size_t STATUS_BYTES = M3SCAN_STATUS_BYTES;

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

struct Plan {
  int B, T, D, K, nc;
  int KS, nsk;  // backward tile (min(K, KT)) and sub-checkpoints per chunk
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
  bool det;              // dB/dC and parameter grads by fixed-order sums of per-block partials
  int dblk;              // channel blocks of the backward's main kernel
  size_t b_dbc;          // workspace offset of those partials [B * T][dblk][2N]
  size_t b_sk;           // workspace offset of the sub-checkpoints [blocks][nsk][N][ch]
  // the split backward over 2..FIN_MAX segments, not deterministic: the
  // segments of a channel block form a cluster that finishes the parameter
  // gradients and d_x at the boundaries itself (no tail kernel)
  bool fin;
};
constexpr int FIN_MAX = 8;  // portable cluster size

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Record a failed CUDA call for m3scan_last_cuda_error (m3_api.cu).
cudaError_t note(cudaError_t e);

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
// The same with clusters of cy blocks along grid y.
template <typename... Args, typename... Vals>
cudaError_t launch_k_cluster_y(void (*kern)(Args...), dim3 grid, unsigned block, size_t smem,
                               cudaStream_t st, bool pdl, unsigned cy, Vals... vals) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = cy;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, vals...);
}

// Fill a tiled tensor map (host; the driver function is found at run time):
// rank 3 or 4, dims innermost first, strides in bytes of dims 1.., box in
// elements; es = 2 (bf16) or 4 (f32).  False if the driver refuses it.
bool encode_tile_map(CUtensorMap* map, int es, int rank, const void* ptr, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);
// Per-unit device status word: nonzero once a kernel of that unit gave up
// waiting for a tile copy.  take_*_status reads and clears it (synchronous).
cudaError_t take_bwd_status(unsigned* out);
cudaError_t take_bwd2_status(unsigned* out);
// the split backward main kernel for (deterministic dB/dC, stop at du,
// carried state, d_state); provided by m3_bwd2.cu
template <typename T> void (*bwd2_kernel_for(bool det, bool scan, bool st, int N))(BwdArgs);
// one block whose tile wait never completes (diagnostic of the bounded waits)
cudaError_t launch_wait_timeout(unsigned* ws_status, cudaStream_t st);
cudaError_t take_fwd_status(unsigned* out);
cudaError_t take_aux_status(unsigned* out);

// Provided by m3_fwd.cu, m3_bwd.cu and m3_aux.cu for T = float and
// __nv_bfloat16.
template <typename T> m3_status launch_fwd(const Plan& p, FwdArgs a, cudaStream_t st);
template <typename T>
m3_status launch_bwd(const Plan& p, BwdArgs a, cudaStream_t st, int smem_per_sm, bool scan);
template <typename T> cudaError_t launch_conv_bwd(ConvArgs a, dim3 grid, cudaStream_t st);
template <typename T> cudaError_t launch_decode_n(int n, const DecArgs& a, cudaStream_t st, int sms);
// kernel attributes (once per device) and occupancy of the one-thread kernels
template <typename T> cudaError_t set_fwd_attrs();
template <typename T> cudaError_t set_bwd_attrs();
template <typename T> cudaError_t set_aux_attrs();
template <typename T> cudaError_t fwd_occupancy(int* blocks);
template <typename T> cudaError_t bwd_occupancy(int chunk, int smem_per_sm, int* blocks);

}  // namespace m3

// m3_bwd.cu -- the backward kernels (segment carries, the one-thread and
// split main kernels, the parameter-gradient tail) and their launch.
#include "m3_common.cuh"

namespace m3 {

// nonzero once a kernel here gave up waiting for a tile copy
__device__ unsigned int g_bwd_status;

cudaError_t take_bwd_status(unsigned* out) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(v));
  if (e == cudaSuccess && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

// Diagnostic: one block raises an mbarrier's transaction count but issues no
// copy, so the phase never completes; the bounded wait must give up and the
// failure must reach the status word, as in the scan kernels.
__global__ void m3_wait_timeout_kernel(unsigned* ws_status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_expect_tx(&bar, 16);
  const bool landed = mbar_wait(&bar, 0);
  if (__syncthreads_or(!landed) && threadIdx.x == 0) report_timeout(&g_bwd_status, ws_status);
}

cudaError_t launch_wait_timeout(unsigned* ws_status, cudaStream_t st) {
  m3_wait_timeout_kernel<<<1, 32, 0, st>>>(ws_status);
  return cudaGetLastError();
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
__global__ void __launch_bounds__(GB) m3_bwd_agg_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int G = GB / TPC;        // channels per block
  constexpr int NL = N / TPC;        // state lanes per thread
  constexpr int TA = TPC == 1 ? TT : TT2;  // staging tile (steps)
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
  const AggSmem L = agg_smem(sizeof(T), N, TA);
  float* fC = reinterpret_cast<float*>(smem + L.fC);
  const int ntiles = (t_end - t_begin + TA - 1) / TA;
  auto tile_start = [&](int i) { return max(t_begin, t_end - (i + 1) * TA); };
  // Tiles of TA rows (the first one, at the segment's start, overlaps rows
  // already covered; only its own rows are read) by tensor-map copies
  // issued by thread 0.
  __shared__ __align__(8) uint64_t tbar[2];  // tile copies into staging buffer 0 / 1
  if (tid == 0) {
    mbar_init(&tbar[0], 1);
    mbar_init(&tbar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  const bool misaligned = (smem_u32(smem) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  const uint32_t tile_bytes = (uint32_t)((3 * TA * G + TA * N) * sizeof(T));
  auto stage = [&](int i, int buf) {
    if (tid == 0 && !misaligned) {
      unsigned char* base = smem + (size_t)buf * L.tile;
      const int t0 = tile_start(i);
      fence_proxy_async();
      mbar_expect_tx(&tbar[buf], tile_bytes);
      tma_load_3d(base + L.dr, &a.tm[TM_ADR], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.z, &a.tm[TM_AZ], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.dg, &a.tm[TM_ADG], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.Ct, &a.tm[TM_AC], 0, t0, b, &tbar[buf]);
    }
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

  if (!a.dbc_part) {
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
    if (a.fin && !a.accumulate) {
      // the main kernel adds its parameter sums into the outputs
      for (size_t i = cid * GB + tid; i < (size_t)g.D * N; i += ncta * GB) a.d_a_log[i] = 0.f;
      for (size_t i = cid * GB + tid; i < (size_t)g.D; i += ncta * GB) {
        a.dD[i] = 0.f;
        a.d_dt_bias[i] = 0.f;
        if (a.d_conv_b) a.d_conv_b[i] = 0.f;
      }
      if (a.d_conv_w)
        for (size_t i = cid * GB + tid; i < (size_t)g.D * WC; i += ncta * GB) a.d_conv_w[i] = 0.f;
    }
  }
  for (int i = 0; i < ntiles; ++i) {
    const int buf = i & 1;
    if (i + 1 < ntiles) stage(i + 1, buf ^ 1);
    const bool landed = !misaligned && mbar_wait(&tbar[buf], (i >> 1) & 1);
    if (__syncthreads_or(!landed)) {
      // a tile did not arrive: report it, let the copy issued above drain, leave
      if (tid == 0) {
        report_timeout(&g_bwd_status, a.status);
        if (!misaligned && i + 1 < ntiles) mbar_wait(&tbar[buf ^ 1], ((i + 1) >> 1) & 1);
      }
      return;
    }
    const unsigned char* base = smem + (size_t)buf * L.tile;
    const int t0 = tile_start(i);
    const int steps = (t_end - i * TA) - t0;
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
      // this thread's NL lanes of C_t, four at a time (16-byte loads)
      const float4* C4 = reinterpret_cast<const float4*>(fC + j * N + NL * hf);
#pragma unroll
      for (int q4 = 0; q4 < NL / 4; ++q4) {
        const float4 cv = C4[q4];
        const int q = 2 * q4;
        carry[q] = __fmul2_rn(ex2x2(__fmul2_rn(dl2, a2[q])),
                              __ffma2_rn(dy2, make_float2(cv.x, cv.y), carry[q]));
        carry[q + 1] = __fmul2_rn(ex2x2(__fmul2_rn(dl2, a2[q + 1])),
                                  __ffma2_rn(dy2, make_float2(cv.z, cv.w), carry[q + 1]));
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

// Sum over the 32 lanes of 16 values held as 8 pairs (element e of pair P:
// state lane 4 * ((P >> 1) ^ (lane & 3)) + 2 * (P & 1) + e); returns the
// total for state lane 4 * (lane & 3) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1).
__device__ __forceinline__ float warp_sum16_rotated(float2 (&v)[NS / 2], int lane) {
  constexpr unsigned FULL = 0xffffffffu;
#pragma unroll
  for (int P = 0; P < 4; ++P)
    v[P] = __fadd2_rn(v[P], make_float2(__shfl_xor_sync(FULL, v[P + 4].x, 2), __shfl_xor_sync(FULL, v[P + 4].y, 2)));
#pragma unroll
  for (int P = 0; P < 2; ++P)
    v[P] = __fadd2_rn(v[P], make_float2(__shfl_xor_sync(FULL, v[P + 2].x, 1), __shfl_xor_sync(FULL, v[P + 2].y, 1)));
  {
    const bool up = (lane & 8) != 0;
    const float2 send = up ? v[0] : v[1];
    const float2 keep = up ? v[1] : v[0];
    v[0] = __fadd2_rn(keep, make_float2(__shfl_xor_sync(FULL, send.x, 8), __shfl_xor_sync(FULL, send.y, 8)));
  }
  const bool up = (lane & 4) != 0;
  const float r = (up ? v[0].y : v[0].x) + __shfl_xor_sync(FULL, up ? v[0].x : v[0].y, 4);
  return r + __shfl_xor_sync(FULL, r, 16);
}

// ST: compiled with the carried-state terms; the plain entry points run the
// instance without them.  SCAN: stop at du (written out) -- the SiLU and
// conv backward then run in m3_conv_bwd_kernel with du plus any gradient
// reaching u from outside the layer core.
//
// Work: a block owns 128 channels of one batch row over one time segment
// (whole chunks of K steps, K the checkpoint interval) and walks its chunks
// last to first.  A chunk is split into tiles of KS = min(K, 8) steps, the
// most whose recomputed states fit the block's tensor memory.  The items of
// chunk c (nt tiles) are, in order:
//   items 0 .. nt-2: tiles 0 .. nt-2 forward from the chunk's checkpoint,
//     leaving the state before tiles 1 .. nt-2 in the workspace (the
//     sub-checkpoints, written with an L2 keep-resident hint: they are read
//     back within the same chunk) and the state before tile nt-1 in the
//     shared memory of the next item;
//   items nt-1 .. 2nt-2: the backward of tiles nt-1 .. 0, each from its
//     start state (the chunk's checkpoint for tile 0).
// Every item's tiles arrive by tensor-map copies into one of two staging
// buffers while the item before runs.  A backward item writes dz, d_delta_raw
// and d_x (du in SCAN mode) into the buffer regions its inputs z, delta_raw
// and d_gated no longer need, and stores them with tile copies.
template <typename T, bool ST, bool SCAN>
__global__ void __launch_bounds__(GB, 3) m3_bwd_kernel(const __grid_constant__ BwdArgs a) {
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
  const int K = g.K, KS = g.KS;
  const BwdSmem L = bwd_smem(KT, sizeof(T));  // laid out for KT-step tiles; a tile may be shorter
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);
  float* red = reinterpret_cast<float*>(smem + L.red);
  // state lane of register slot 2*i (pair i): quad (i >> 1) ^ rot, offset 2*(i & 1)
  auto lane_of = [&](int i) { return 4 * ((i >> 1) ^ rot) + 2 * (i & 1); };
  // this thread's quads of a row of B or C, in register order
  const float4* fBq[4];
  const float4* fCq[4];
#pragma unroll
  for (int qs = 0; qs < 4; ++qs) {
    fBq[qs] = reinterpret_cast<const float4*>(fB) + (qs ^ rot);
    fCq[qs] = reinterpret_cast<const float4*>(fC) + (qs ^ rot);
  }
  // this block's sub-checkpoint slot in the workspace
  auto slot = [&]() { return (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)); };

  // The recomputed states of a tile (KS rows of 16 f32 per channel) live in
  // tensor memory: row j of this thread = columns [16 j, 16 j + 16) of its
  // lane.  Warp 0 allocates for the CTA; every exit path below deallocates.
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t tbar[2];  // tile copies into staging buffer 0 / 1
  if (warp == 0) tmem_alloc(&tmem_slot, a.tcols);
  if (tid == 32) {
    mbar_init(&tbar[0], 1);
    mbar_init(&tbar[1], 1);
    mbar_init_fence();
  }
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
  // The tiles of an item arrive by tensor-map copies issued by thread 0: x
  // with its three halo rows before the tile, delta_raw and B; for a
  // backward item also z, d_gated and C; and the start state (16 rows of GB
  // floats) when it comes from the chunk's checkpoint or a sub-checkpoint.
  // Rows outside [0, T) and channels past d_inner arrive as zeros.
  // tiles of chunk c: one when a chunk is at most a tile, else whole KT-step
  // tiles (a shift, no division)
  auto tiles_of = [&](int c) { return K <= KT ? 1 : (min(K, g.T - c * K) + KT - 1) / KT; };
  const bool misaligned = (smem_u32(smem) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  auto stage = [&](int c, int q, int buf) {
    if (tid == 0 && !misaligned) {
      const uint32_t fwd_bytes = (uint32_t)(((2 * KS + 3) * GB + KS * NS) * sizeof(T));
      const uint32_t bwd_bytes = (uint32_t)(((4 * KS + 3) * GB + 2 * KS * NS) * sizeof(T));
      const uint32_t ck_bytes = (uint32_t)(NS * GB * 4);
      const int nt = tiles_of(c);
      const bool fw = q < nt - 1;
      const int j = fw ? q : 2 * nt - 2 - q;
      const int t0 = c * K + j * KS;
      const bool ck_chunk = j == 0;
      const bool ck_sub = !fw && j >= 1 && j <= nt - 2;
      unsigned char* base = smem + (size_t)buf * L.tile;
      // the tile stores of the item that last used this buffer have read it
      bulk_wait_read();
      fence_proxy_async();
      mbar_expect_tx(&tbar[buf], (fw ? fwd_bytes : bwd_bytes) + (ck_chunk || ck_sub ? ck_bytes : 0u));
      tma_load_3d(base + L.x, &a.tm[TM_X], d0, t0 - 3, b, &tbar[buf]);
      tma_load_3d(base + L.dr, &a.tm[TM_DR], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.Bt, &a.tm[TM_B], 0, t0, b, &tbar[buf]);
      if (!fw) {
        tma_load_3d(base + L.z, &a.tm[TM_Z], d0, t0, b, &tbar[buf]);
        tma_load_3d(base + L.dg, &a.tm[TM_DG], d0, t0, b, &tbar[buf]);
        tma_load_3d(base + L.Ct, &a.tm[TM_C], 0, t0, b, &tbar[buf]);
      }
      if (ck_chunk) tma_load_4d(base + L.ck, &a.tm[TM_CK], d0, 0, c, b, &tbar[buf]);
      if (ck_sub) tma_load_4d(base + L.ck, &a.tm[TM_SK], 0, 0, j - 1, slot(), &tbar[buf]);
    }
  };

  if (c_begin < c_end) stage(c_end - 1, 0, 0);  // first item in flight while the carries load
  grid_dep_trigger();
  // the aggregate kernel's carries, and its clearing of dB and dC before
  // this kernel's reductions into them
  grid_dep_wait();
  if (s + 1 < g.S) {
    // chain the later segments right to left: in(s'-1) = exp(A sum delta_s')
    // in(s') + local(s'), with in(S-1) = 0
    chain_segments<NS / 2, 2>(carry, a2, a.sd, a.q, NS, (size_t)b * g.S, g.S - 1, -1, g.S - 1 - s,
                              g.D, d, active, lane_of);
  }
  float2 dAp[NS / 2];  // dL/dA per lane
#pragma unroll
  for (int i = 0; i < NS / 2; ++i) dAp[i] = make_float2(0.f, 0.f);
  float dD_acc = 0.f, ddtb_acc = 0.f, dcb_acc = 0.f;
  float dcw[WC] = {0.f, 0.f, 0.f, 0.f};
  float dc1 = 0.f, dc2 = 0.f, dc3 = 0.f;  // conv-input gradient at t+1, t+2, t+3

  bool aborted = false;
  int it = 0;  // items so far: buffer it & 1, its (it >> 1)-th use
  for (int c = c_end - 1; c >= c_begin && !aborted; --c) {
    const int nt = tiles_of(c);
    const int nq = 2 * nt - 1;
    for (int q = 0; q < nq; ++q, ++it) {
      const int buf = it & 1;
      const bool more = q + 1 < nq || c - 1 >= c_begin;
      const bool fw = q < nt - 1;
      // The next item's tiles: a forward item issues them now; a backward
      // item after its first scalar pass, by when the tile stores of the item
      // before (which read the buffer being refilled) have long finished.
      auto stage_next = [&]() {
        if (q + 1 < nq) stage(c, q + 1, buf ^ 1);
        else if (c - 1 >= c_begin) stage(c - 1, 0, buf ^ 1);
      };
      if (fw) stage_next();
      const bool landed = !misaligned && mbar_wait(&tbar[buf], (it >> 1) & 1);
      if (__syncthreads_or(!landed)) {
        // a tile did not arrive: report it, let a copy issued above drain, leave
        if (tid == 0) {
          report_timeout(&g_bwd_status, a.status);
          if (!misaligned && fw && more) mbar_wait(&tbar[buf ^ 1], ((it + 1) >> 1) & 1);
        }
        aborted = true;
        break;
      }
      const int j = fw ? q : 2 * nt - 2 - q;  // tile within the chunk
      const int t0 = c * K + j * KS;          // its first step
      const int steps = min(KS, min(c * K + K, g.T) - t0);
      unsigned char* base = smem + (size_t)buf * L.tile;
      if (ST && a.conv_in && t0 < 3 && active) {
        // halo rows before step 0 (staged as zeros): the carried conv inputs.
        // Only this thread reads its column of the x tile.
        T* xw = reinterpret_cast<T*>(base + L.x);
        const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * g.D + d;
        for (int r = 0; r < 3 - t0; ++r) xw[r * GB + tid] = ci[(size_t)(t0 + r) * g.D];
      }
      {
        const T* Bt = reinterpret_cast<const T*>(base + L.Bt);
        const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
        for (int i = tid; i < KS * NS; i += GB) {
          fB[i] = Act<T>::ld(Bt + i);
          if (!fw) fC[i] = Act<T>::ld(Ct + i);
        }
      }
      __syncthreads();
      const T* xt = reinterpret_cast<const T*>(base + L.x);  // row r is step t0 - 3 + r
      const T* drt = reinterpret_cast<const T*>(base + L.dr);
      float* ckt = reinterpret_cast<float*>(base + L.ck);
      float4* s0 = reinterpret_cast<float4*>(smem + L.scal) + tid;  // thread-private, stride GB
      float4* s1 = s0 + (size_t)KT * GB;

      if (fw) {
        // ---- forward item: the states through tile j, from the start state
        // in this buffer (the chunk's checkpoint for tile 0, else left by the
        // forward item before) ----
        float2 hs[NS / 2];
#pragma unroll
        for (int i = 0; i < NS / 2; ++i) {
          const int n = lane_of(i);
          hs[i] = make_float2(ckt[n * GB + tid], ckt[(n + 1) * GB + tid]);
        }
        {
          float xm3 = Act<T>::ld(xt + 0 * GB + tid);
          float xm2 = Act<T>::ld(xt + 1 * GB + tid);
          float xm1 = Act<T>::ld(xt + 2 * GB + tid);
#pragma unroll
          for (int jj = 0; jj < KT; ++jj) {
            if (jj >= steps) break;
            const float xv = Act<T>::ld(xt + (jj + 3) * GB + tid);
            const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
            xm3 = xm2;
            xm2 = xm1;
            xm1 = xv;
            const float u = cpre * sigmoid_f(cpre);
            const float delta = softplus_f(Act<T>::ld(drt + jj * GB + tid) + dtb);
            *reinterpret_cast<float2*>(s0 + jj * GB) = make_float2(delta, delta * u);
          }
        }
#pragma unroll
        for (int jj = 0; jj < KT; ++jj) {
          if (jj >= steps) break;
          const float2 v0 = *reinterpret_cast<const float2*>(s0 + jj * GB);
          const float2 dl2 = f2b(v0.x);
          const float2 du2 = f2b(v0.y);
#pragma unroll
          for (int qs = 0; qs < 4; ++qs) {
            const float4 bv = fBq[qs][jj * (NS / 4)];
            hs[2 * qs] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[2 * qs])), hs[2 * qs],
                                    __fmul2_rn(du2, make_float2(bv.x, bv.y)));
            hs[2 * qs + 1] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[2 * qs + 1])), hs[2 * qs + 1],
                                        __fmul2_rn(du2, make_float2(bv.z, bv.w)));
          }
        }
        if (j + 1 < nt - 1) {
          // the state before tile j + 1: a sub-checkpoint, read back by the
          // backward item of that tile with a tile copy
          float* skp = a.sk + ((size_t)slot() * g.nsk + j) * NS * GB + tid;
          const uint64_t keep_policy = l2_evict_last_policy();
#pragma unroll
          for (int i = 0; i < NS / 2; ++i) {
            const int n = lane_of(i);
            st_keep(skp + n * GB, hs[i].x, keep_policy);
            st_keep(skp + (n + 1) * GB, hs[i].y, keep_policy);
          }
          fence_proxy_async_global();
        }
        {
          // and the start state of the next item (the next forward item, or
          // the backward item of the last tile), whose copies bring none
          float* ckn = reinterpret_cast<float*>(smem + (size_t)(buf ^ 1) * L.tile + L.ck);
#pragma unroll
          for (int i = 0; i < NS / 2; ++i) {
            const int n = lane_of(i);
            ckn[n * GB + tid] = hs[i].x;
            ckn[(n + 1) * GB + tid] = hs[i].y;
          }
        }
        __syncthreads();
        continue;
      }

      // ---- backward item: tile j ----
      const T* zt = reinterpret_cast<const T*>(base + L.z);
      const T* dgt = reinterpret_cast<const T*>(base + L.dg);
      // outputs, staged where the inputs no longer needed were: dz over z,
      // d_delta_raw over delta_raw, d_x (or du when stopping at du) over d_gated
      T* oz = reinterpret_cast<T*>(base + L.z);
      T* odr = reinterpret_cast<T*>(base + L.dr);
      T* odx = reinterpret_cast<T*>(base + L.dg);
      T* const du_c = (!SCAN && a.du_dbg)
                          ? static_cast<T*>(a.du_dbg) + ((size_t)b * g.T + (size_t)t0) * g.D + d
                          : nullptr;
      const int nst = steps;

      // ---- scalar pass: everything per step that does not need the state ----
      {
        float xm3 = Act<T>::ld(xt + 0 * GB + tid);
        float xm2 = Act<T>::ld(xt + 1 * GB + tid);
        float xm1 = Act<T>::ld(xt + 2 * GB + tid);
#pragma unroll 2
        for (int jj = 0; jj < KT; ++jj) {
          if (jj >= nst) break;
          const float xv = Act<T>::ld(xt + (jj + 3) * GB + tid);
          const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
          xm3 = xm2;
          xm2 = xm1;
          xm1 = xv;
          const float sc = sigmoid_f(cpre);
          const float u = cpre * sc;
          const float2 sps = softplus_sigmoid(Act<T>::ld(drt + jj * GB + tid) + dtb);
          const float delta = sps.x;
          const float zv = Act<T>::ld(zt + jj * GB + tid);
          const float gv = Act<T>::ld(dgt + jj * GB + tid);
          const float sz = sigmoid_f(zv);
          const float dy = gv * zv * sz;                           // dL/dy
          const float dzf = gv * (sz * fmaf(zv, 1.f - sz, 1.f));    // dL/dz = y * dzf
          s0[jj * GB] = make_float4(delta, delta * u, dy, dzf);
          s1[jj * GB] = make_float4(Dd * u, sps.y, sc, cpre);
        }
      }

      stage_next();

      // ---- recompute the tile's states from its start state ----
      {
        float2 h[NS / 2];
#pragma unroll
        for (int i = 0; i < NS / 2; ++i) {
          const int n = lane_of(i);
          h[i] = make_float2(ckt[n * GB + tid], ckt[(n + 1) * GB + tid]);
        }
#pragma unroll
        for (int jj = 0; jj < KT; ++jj) {
          if (jj >= nst) break;
          const float2 v0 = *reinterpret_cast<const float2*>(s0 + jj * GB);
          const float2 dl2 = f2b(v0.x);
          const float2 du2 = f2b(v0.y);
#pragma unroll
          for (int qs = 0; qs < 4; ++qs) {
            const float4 bv = fBq[qs][jj * (NS / 4)];
            const float2 dA0 = ex2x2(__fmul2_rn(dl2, a2[2 * qs]));
            const float2 dA1 = ex2x2(__fmul2_rn(dl2, a2[2 * qs + 1]));
            h[2 * qs] = __ffma2_rn(dA0, h[2 * qs], __fmul2_rn(du2, make_float2(bv.x, bv.y)));
            h[2 * qs + 1] = __ffma2_rn(dA1, h[2 * qs + 1], __fmul2_rn(du2, make_float2(bv.z, bv.w)));
          }
          tmem_st16(trow + 16u * (uint32_t)jj, h);
        }
        tmem_wait_st();
      }

      // ---- reverse-time pass: y and dz, adjoint state, dA, dB/dC ----
      {
        // this lane's row of the dB/dC sums: lanes 0-15 dB, 16-31 dC
        float* const red_l = red + warp * 32 +
                             (lane < 16 ? 0 : 16) + 4 * rot + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
        // One step: hn = h_t (state after step t = jj), hp receives h_{t-1}.
        auto rev_step = [&](const int jj, const float2 (&hn)[NS / 2], float2 (&hp)[NS / 2]) {
          const float4 v0 = s0[jj * GB];
          const float Du = reinterpret_cast<const float*>(s1 + jj * GB)[0];
          const float2 dl2 = f2b(v0.x);
          const float2 du2 = f2b(v0.y);
          const float2 dy2 = f2b(v0.z);
          float2 sB = make_float2(0.f, 0.f), sAq = make_float2(0.f, 0.f);
          float2 y01 = make_float2(0.f, 0.f), y23 = make_float2(0.f, 0.f);
          float2 pB[NS / 2], pC[NS / 2];
          if (jj > 0) {
            tmem_ld16(trow + 16u * (uint32_t)(jj - 1), hp);
          } else {
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) {
              const int n = lane_of(i);
              hp[i] = make_float2(ckt[n * GB + tid], ckt[(n + 1) * GB + tid]);
            }
          }
#pragma unroll
          for (int qs = 0; qs < 4; ++qs) {
            const float4 bv = fBq[qs][jj * (NS / 4)];
            const float4 cv = fCq[qs][jj * (NS / 4)];
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
          const float y = ((y01.x + y01.y) + (y23.x + y23.y)) + Du;
          Act<T>::st(oz + jj * GB + tid, y * v0.w);
          // the scalar pass below reads these two sums
          reinterpret_cast<float*>(s0 + jj * GB)[3] = sAq.x + sAq.y;
          reinterpret_cast<float*>(s1 + jj * GB)[0] = sB.x + sB.y;
          // Channels past d_inner run on zero-filled inputs and parameters, so
          // their partials are exactly zero and need no masking.
          const float rb = warp_sum16_rotated(pB, lane);
          const float rc = warp_sum16_rotated(pC, lane);
          red_l[jj * NWB * 32] = lane < 16 ? rb : rc;
        };
        float2 hA[NS / 2], hB[NS / 2];
        tmem_ld16(trow + 16u * (uint32_t)(nst - 1), hA);
        if (nst == KT) {
          // a whole tile: steps in pairs, the two state registers trading roles
#pragma unroll 1
          for (int jj = KT - 1; jj > 0; jj -= 2) {
            rev_step(jj, hA, hB);
            rev_step(jj - 1, hB, hA);
          }
        } else {
#pragma unroll 1
          for (int jj = nst - 1; jj >= 0; --jj) {
            rev_step(jj, hA, hB);
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) hA[i] = hB[i];
          }
        }
      }

      // ---- scalar pass: du, d delta, softplus, SiLU and conv backward ----
      // conv inputs of steps t-2, t-1, t (tile rows j+1 .. j+3), slid down a row per step
      float xw1 = Act<T>::ld(xt + nst * GB + tid), xw2 = Act<T>::ld(xt + (nst + 1) * GB + tid),
            xw3 = Act<T>::ld(xt + (nst + 2) * GB + tid);
      // whether any step of this tile writes the optional du, or a segment
      // boundary term (one test per tile instead of per step)
      const bool edge = du_c != nullptr || (s + 1 < g.S && t0 + nst > t_end - 3) ||
                        (s > 0 && t0 < t_begin + 3);
#pragma unroll 2
      for (int jj = KT - 1; jj >= 0; --jj) {
        if (jj >= nst) continue;
        const int t = t0 + jj;
        const float4 v0 = s0[jj * GB];
        const float4 v1 = s1[jj * GB];
        const float delta = v0.x, dy = v0.z, sAq = v0.w;
        const float sumB = v1.x, sv = v1.y, sc = v1.z, cpre = v1.w;
        const float u = cpre * sc;
        const float du = fmaf(dy, Dd, delta * sumB);
        const float ddr = fmaf(u, sumB, LN2 * sAq) * sv;
        dD_acc = fmaf(dy, u, dD_acc);
        ddtb_acc += ddr;
        Act<T>::st(odr + jj * GB + tid, ddr);
        if constexpr (SCAN) {  // the SiLU and conv backward run later, with du
          Act<T>::st(odx + jj * GB + tid, du);
          continue;
        }
        const float dc = du * (sc * fmaf(cpre, 1.f - sc, 1.f));
        dcb_acc += dc;
        const float xw0 = Act<T>::ld(xt + jj * GB + tid);
        dcw[0] = fmaf(dc, xw0, dcw[0]);
        dcw[1] = fmaf(dc, xw1, dcw[1]);
        dcw[2] = fmaf(dc, xw2, dcw[2]);
        dcw[3] = fmaf(dc, xw3, dcw[3]);
        xw3 = xw2;
        xw2 = xw1;
        xw1 = xw0;
        float dxv = fmaf(dc, w[3], fmaf(dc1, w[2], fmaf(dc2, w[1], dc3 * w[0])));
        if (ST && a.g_conv && t >= g.T - 3 && active)  // x[t] is also a conv-state output
          dxv += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + t - (g.T - 3)) * g.D + d);
        dc3 = dc2;
        dc2 = dc1;
        dc1 = dc;
        // at the last three steps before a later segment d_x still lacks that
        // segment's terms: the tail kernel writes those rows again, complete
        Act<T>::st(odx + jj * GB + tid, dxv);
        if (edge && active) {
          if (du_c) Act<T>::st(du_c + (size_t)jj * g.D, du);
          if (s + 1 < g.S && t >= t_end - 3)
            a.dxpart[(((size_t)b * g.S + s) * 3 + (t - (t_end - 3))) * g.D + d] = dxv;
          if (s > 0 && t < t_begin + 3)
            a.dchead[(((size_t)b * g.S + s) * 3 + (t - t_begin)) * g.D + d] = dc;
        }
      }

      fence_proxy_async();  // this thread's output rows, before the tile stores read them
      __syncthreads();
      if (tid == 0) {
        // rows past the sequence and channels past d_inner are not written
        tma_store_3d(&a.tm[TM_ODZ], oz, d0, t0, b);
        tma_store_3d(&a.tm[TM_ODR], odr, d0, t0, b);
        tma_store_3d(&a.tm[SCAN ? TM_ODU : TM_ODX], odx, d0, t0, b);
        bulk_commit();
      }
      // one global reduction per (t, n) per block for dB and dC
      if (a.dbc_part) {  // this block's share, summed in a fixed order by m3_dbc_sum_kernel
        for (int i = tid; i < steps * 32; i += GB) {
          const int jj = i >> 5, l = i & 31;
          float v = 0.f;
#pragma unroll
          for (int ww = 0; ww < NWB; ++ww) v += red[(jj * NWB + ww) * 32 + l];
          a.dbc_part[(((size_t)b * g.T + t0 + jj) * a.nblk + blockIdx.x) * 32 + l] = v;
        }
      } else {
        for (int i = tid; i < steps * 32; i += GB) {
          const int jj = i >> 5, l = i & 31;
          float v = 0.f;
#pragma unroll
          for (int ww = 0; ww < NWB; ++ww) v += red[(jj * NWB + ww) * 32 + l];
          float* dst = (l < NS ? a.dB : a.dC) + ((size_t)b * g.T + t0 + jj) * g.lddbc + (l & (NS - 1));
          atomicAdd(dst, v);
        }
      }
      __syncthreads();
    }
  }

  if (!aborted) {
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
  }
  if (tid == 0) bulk_wait_all();  // the tile stores are done before the block's memory goes
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_slot, a.tcols);
}

// Deterministic dB/dC (launched after the main kernel when asked for): the
// channel blocks' shares of one (batch, step, lane) summed in block order.
__global__ void m3_dbc_sum_kernel(BwdArgs a, int N) {
  const Geo g = a.g;
  grid_dep_wait();  // the main kernel's shares
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t bt = idx / (2 * N);
  const int l = (int)(idx % (2 * N));
  if (bt >= (size_t)g.B * g.T) return;
  const float* p = a.dbc_part + bt * a.nblk * 2 * N + l;
  float v = 0.f;
  for (int k = 0; k < a.nblk; ++k) v += p[(size_t)k * 2 * N];
  (l < N ? a.dB : a.dC)[bt * g.lddbc + (l % N)] = v;
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
__global__ void m3_bwd_tail_kernel(TailArgs a, int rows, int nfin, int nout, int N) {
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

template <typename T>
void (*agg_for(bool split, int N))(BwdArgs) {
  if (!split) return m3_bwd_agg_kernel<T, 1, 16>;
  return N == 16 ? m3_bwd_agg_kernel<T, 2, 16>
       : N == 32 ? m3_bwd_agg_kernel<T, 4, 32> : m3_bwd_agg_kernel<T, 8, 64>;
}

// scan: stop at du (m3scan_bwd_scan); the conv side runs in launch_conv_bwd.
// Tensor maps of the backward's tiles (boxes of ch channels).
template <typename T>
bool encode_bwd_maps(const Plan& p, int ch, bool scan, BwdArgs& a) {
  const uint64_t es = sizeof(T), D = p.D, T_ = p.T, B = p.B, N = p.N, ld = p.ldbc, nc = p.nc;
  const uint32_t K = (uint32_t)p.KS, c = (uint32_t)ch, n = (uint32_t)p.N;  // tiles of KS steps
  const uint64_t adim[3] = {D, T_, B}, astr[2] = {D * es, T_ * D * es};
  const uint64_t bdim[3] = {N, T_, B}, bstr[2] = {ld * es, T_ * ld * es};
  const uint64_t cdim[4] = {D, N, nc, B}, cstr[3] = {D * 4, N * D * 4, nc * N * D * 4};
  const uint32_t box_x[3] = {c, K + 3, 1}, box_a[3] = {c, K, 1}, box_b[3] = {n, K, 1}, box_c[4] = {c, n, 1, 1};
  const uint32_t ta = (uint32_t)(p.bwd_tpc == 1 ? TT : TT2);  // the aggregate kernel's tile
  const uint32_t box_ta[3] = {c, ta, 1}, box_tb[3] = {n, ta, 1};
  bool ok = true;
  if (p.nsk > 0) {  // sub-checkpoints [blocks][nsk][N][ch]
    const uint64_t blocks = (uint64_t)((p.D + ch - 1) / ch) * p.Sb * p.B, nsk = p.nsk;
    const uint64_t sdim[4] = {(uint64_t)ch, N, nsk, blocks};
    const uint64_t sstr[3] = {(uint64_t)ch * 4, N * ch * 4, nsk * N * ch * 4};
    ok = encode_tile_map(&a.tm[TM_SK], 4, 4, a.sk, sdim, sstr, box_c);
  }
  if (p.bwd_tpc == 1) {  // the one-thread kernel stores its tiles of dz, d_delta_raw, d_x / du
    ok = ok && encode_tile_map(&a.tm[TM_ODZ], (int)es, 3, a.dz, adim, astr, box_a) &&
         encode_tile_map(&a.tm[TM_ODR], (int)es, 3, a.ddr, adim, astr, box_a) &&
         (scan ? encode_tile_map(&a.tm[TM_ODU], (int)es, 3, a.du_dbg, adim, astr, box_a)
               : encode_tile_map(&a.tm[TM_ODX], (int)es, 3, a.dx, adim, astr, box_a));
  }
  ok = ok && encode_tile_map(&a.tm[TM_X], (int)es, 3, a.x, adim, astr, box_x) &&
                  encode_tile_map(&a.tm[TM_DR], (int)es, 3, a.dr, adim, astr, box_a) &&
                  encode_tile_map(&a.tm[TM_Z], (int)es, 3, a.z, adim, astr, box_a) &&
                  encode_tile_map(&a.tm[TM_DG], (int)es, 3, a.dg, adim, astr, box_a) &&
                  encode_tile_map(&a.tm[TM_B], (int)es, 3, a.Bm, bdim, bstr, box_b) &&
                  encode_tile_map(&a.tm[TM_C], (int)es, 3, a.Cm, bdim, bstr, box_b) &&
                  encode_tile_map(&a.tm[TM_CK], 4, 4, a.ckpt, cdim, cstr, box_c) &&
                  encode_tile_map(&a.tm[TM_ADR], (int)es, 3, a.dr, adim, astr, box_ta) &&
                  encode_tile_map(&a.tm[TM_AZ], (int)es, 3, a.z, adim, astr, box_ta) &&
                  encode_tile_map(&a.tm[TM_ADG], (int)es, 3, a.dg, adim, astr, box_ta) &&
                  encode_tile_map(&a.tm[TM_AC], (int)es, 3, a.Cm, bdim, bstr, box_tb);
  if (!ok) note(cudaErrorInvalidValue);
  return ok;
}

template <typename T>
m3_status launch_bwd(const Plan& p, BwdArgs a, cudaStream_t st, int smem_per_sm, bool scan) {
  const int groups = (p.D + GB - 1) / GB;
  a.g = Geo{p.B, p.T, p.D, p.K, p.nc, p.Sb, p.mb, p.ldbc, p.lddbc, p.KS, p.nsk};
  cudaError_t e = cudaSuccess;
  if (!encode_bwd_maps<T>(p, p.bwd_tpc != 1 ? 128 / (p.N / 8) : GB, scan, a)) return M3_ERR_CUDA;
  if (p.Sb > 1) {
    // also clears dB and dC before the main kernel's reductions into them
    const bool split = p.bwd_tpc != 1;
    const int ch = split ? 128 / (p.N / 8) : GB;
    e = launch_k(agg_for<T>(split, p.N), dim3((p.D + ch - 1) / ch, p.Sb - 1, p.B), GB,
                 agg_smem(sizeof(T), p.N, split ? TT2 : TT).total, st, false, a);
    if (note(e) != cudaSuccess) return M3_ERR_CUDA;
  } else if (!p.det) {
    // only the d_state columns of each (batch, step) row belong to dB and dC
    const size_t pitch = (size_t)p.lddbc * 4, rows = (size_t)p.B * p.T;
    if (note(cudaMemset2DAsync(a.dB, pitch, 0, (size_t)p.N * 4, rows, st)) != cudaSuccess) return M3_ERR_CUDA;
    if (note(cudaMemset2DAsync(a.dC, pitch, 0, (size_t)p.N * 4, rows, st)) != cudaSuccess) return M3_ERR_CUDA;
  }
  const bool with_state = a.conv_in || a.g_h || a.g_conv || a.d_h_in || a.d_conv_in;
  if (p.bwd_tpc != 1) {
    a.tcols = tmem_cols2_for(KT);
    const size_t smem = bwd2_launch_smem(KT, sizeof(T), p.N, smem_per_sm);
    void (*kern)(BwdArgs) = bwd2_kernel_for<T>(p.det, scan, with_state, p.N);
    const int ch = 128 / (p.N / 8);
    const dim3 grid((p.D + ch - 1) / ch, p.Sb, p.B);
    e = a.fin ? launch_k_cluster_y(kern, grid, 128, smem, st, true, (unsigned)p.Sb, a)
              : launch_k(kern, grid, 128, smem, st, p.Sb > 1, a);
  } else {
    a.tcols = tmem_cols_for(KT);
    const size_t smem = bwd_launch_smem(KT, sizeof(T), smem_per_sm);
    void (*kern)(BwdArgs) = scan ? (with_state ? m3_bwd_kernel<T, true, true> : m3_bwd_kernel<T, false, true>)
                                 : (with_state ? m3_bwd_kernel<T, true, false> : m3_bwd_kernel<T, false, false>);
    e = launch_k(kern, dim3(groups, p.Sb, p.B), GB, smem, st, p.Sb > 1, a);
  }
  // parameter outputs: N d_a_log, dD, d_dt_bias (+ d_conv_b, 4 d_conv_w)
  const int nout = scan ? p.N + 2 : p.N + 7;
  const size_t nfin = ((size_t)nout * p.D + 31) / 32;                 // 32 outputs per block
  const size_t nfix = (!scan && p.Sb > 1) ? ((size_t)p.B * (p.Sb - 1) * 3 * p.D + 255) / 256 : 0;
  const size_t ndbc = p.det ? ((size_t)p.B * p.T * 2 * p.N + 255) / 256 : 0;
  if (e == cudaSuccess && !a.fin) {
    TailArgs ta;
    ta.g = a.g;
    ta.partials = a.partials; ta.dxpart = a.dxpart; ta.dchead = a.dchead;
    ta.conv_w = a.conv_w; ta.a_log = a.a_log; ta.dx = a.dx;
    ta.d_a_log = a.d_a_log; ta.dD = a.dD; ta.d_dt_bias = a.d_dt_bias;
    ta.d_conv_b = a.d_conv_b; ta.d_conv_w = a.d_conv_w; ta.accumulate = a.accumulate;
    e = launch_k(m3_bwd_tail_kernel<T>, dim3((unsigned)(nfin + nfix)), 256, 0, st, true, ta,
                 p.B * p.Sb, (int)nfin, nout, p.N);
  }
  if (e == cudaSuccess && p.det)
    e = launch_k(m3_dbc_sum_kernel, dim3((unsigned)ndbc), 256, 0, st, true, a, p.N);
  if (e == cudaSuccess) e = cudaGetLastError();
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

template <typename T>
cudaError_t set_bwd_attrs() {
  const int es = sizeof(T);
  cudaError_t e = cudaSuccess;
  const bool splits[4] = {false, true, true, true};
  const int ns[4] = {16, 16, 32, 64};
  for (int i = 0; i < 4; ++i) {
    void (*k)(BwdArgs) = agg_for<T>(splits[i], ns[i]);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)agg_smem(es, ns[i], splits[i] ? TT2 : TT).total);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  void (*bwd_kernels[28])(BwdArgs) = {
      m3_bwd_kernel<T, false, false>, m3_bwd_kernel<T, true, false>, m3_bwd_kernel<T, false, true>,
      m3_bwd_kernel<T, true, true>};
  int nk = 4;
  for (int N : {16, 32, 64})
    for (int v = 0; v < 8; ++v)
      bwd_kernels[nk++] = bwd2_kernel_for<T>(v & 4, v & 1, v & 2, N);
  for (auto k : bwd_kernels) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_CAP);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  }
  return e;
}

template <typename T>
cudaError_t bwd_occupancy(int chunk, int smem_per_sm, int* blocks) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, m3_bwd_kernel<T, false, false>, GB,
                                                       bwd_launch_smem(chunk, sizeof(T), smem_per_sm));
}

template m3_status launch_bwd<float>(const Plan&, BwdArgs, cudaStream_t, int, bool);
template m3_status launch_bwd<__nv_bfloat16>(const Plan&, BwdArgs, cudaStream_t, int, bool);
template cudaError_t set_bwd_attrs<float>();
template cudaError_t set_bwd_attrs<__nv_bfloat16>();
template cudaError_t bwd_occupancy<float>(int, int, int*);
template cudaError_t bwd_occupancy<__nv_bfloat16>(int, int, int*);

}  // namespace m3

// m3_bwd2.cu -- the backward main kernel with the lanes split over
// d_state / 8 threads per channel, compiled apart from the rest of the
// backward so the two build in parallel.
#include "m3_common.cuh"

namespace m3 {

// nonzero once a kernel here gave up waiting for a tile copy
__device__ unsigned int g_bwd2_status;

cudaError_t take_bwd2_status(unsigned* out) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd2_status, sizeof(v));
  if (e == cudaSuccess && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_bwd2_status, &zero, sizeof(zero));
  }
  *out = v;
  return e;
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

template <typename T, bool ST, bool SCAN, int N, bool DET>
__global__ void __launch_bounds__(128, 4) m3_bwd2_kernel(const __grid_constant__ BwdArgs a) {
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
  const int K = g.K, KS = g.KS;  // checkpoint interval; tile
  const Bwd2Smem L = bwd2_smem(KT, sizeof(T), N);  // laid out for KT-step tiles; a tile may be shorter
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);
  float* red = reinterpret_cast<float*>(smem + L.red);
  float* dcs = reinterpret_cast<float*>(smem + L.dcs);  // [KT + 3][CH]
  // state lane of register pair P
  auto lane_of = [&](int P) { return 8 * hf + 2 * (P ^ prot); };
  // this thread's copy of B and C: its 8 lanes in register order
  const float* fBr = fB + prot * rot_stride(KT, N) + 8 * hf;
  const float* fCr = fC + prot * rot_stride(KT, N) + 8 * hf;
  // this block's sub-checkpoint slot in the workspace
  const int slot = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);

  // recomputed states of a chunk: row j of this thread = TMEM columns
  // [8 j, 8 j + 8) of its lane; warp 0 allocates, every exit deallocates
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
  // Work items as in m3_bwd_kernel: for chunk c of nt tiles of KS steps,
  // items 0 .. nt-2 run tiles 0 .. nt-2 forward from the chunk's checkpoint
  // (sub-checkpoints of tiles 1 .. nt-2 to the workspace, the state before
  // tile nt-1 to the next item's staging buffer), items nt-1 .. 2nt-2 the
  // backward of tiles nt-1 .. 0.  An item's tiles arrive by tensor-map copies
  // issued by thread 0: x with its three halo rows, delta_raw, B; for a
  // backward item also z, d_gated, C; and the start state when it comes
  // from the chunk's checkpoint or a sub-checkpoint.  Rows outside [0, T)
  // and channels past d_inner arrive as zeros.
  // tiles of chunk c: one when a chunk is at most a tile, else whole KT-step
  // tiles (a shift, no division)
  auto tiles_of = [&](int c) { return K <= KT ? 1 : (min(K, g.T - c * K) + KT - 1) / KT; };
  const uint32_t fwd_bytes = (uint32_t)(((2 * KS + 3) * CH + KS * N) * sizeof(T));
  const uint32_t bwd_bytes = (uint32_t)(((4 * KS + 3) * CH + 2 * KS * N) * sizeof(T));
  const uint32_t ck_bytes = (uint32_t)(N * CH * 4);
  const bool misaligned = (smem_u32(smem) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  auto stage = [&](int c, int q, int buf) {
    if (tid == 0 && !misaligned) {
      const int nt = tiles_of(c);
      const bool fw = q < nt - 1;
      const int j = fw ? q : 2 * nt - 2 - q;
      const int t0 = c * K + j * KS;
      const bool ck_chunk = j == 0;
      const bool ck_sub = !fw && j >= 1 && j <= nt - 2;
      unsigned char* base = smem + (size_t)buf * L.tile;
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
      if (ck_sub) tma_load_4d(base + L.ck, &a.tm[TM_SK], 0, 0, j - 1, slot, &tbar[buf]);
    }
  };
  if (c_begin < c_end) stage(c_end - 1, 0, 0);
  grid_dep_trigger();
  grid_dep_wait();
  if (s + 1 < g.S) {
    chain_segments<4, 4>(carry, a2, a.sd, a.q, N, (size_t)b * g.S, g.S - 1, -1, g.S - 1 - s, g.D, d,
                         active, lane_of);
  }
  float2 dAp[4];
#pragma unroll
  for (int P = 0; P < 4; ++P) dAp[P] = make_float2(0.f, 0.f);
  float dD_acc = 0.f, ddtb_acc = 0.f, dcb_acc = 0.f;
  float dcw[WC] = {0.f, 0.f, 0.f, 0.f};
  for (int i = tid; i < (KT + 3) * CH; i += 128) dcs[i] = 0.f;  // ordered by the loop's first barrier

  bool aborted = false;
  int it = 0;  // items so far: buffer it & 1, its (it >> 1)-th use
  for (int c = c_end - 1; c >= c_begin && !aborted; --c) {
   const int nt = tiles_of(c);
   const int nq = 2 * nt - 1;
   for (int q = 0; q < nq; ++q, ++it) {
    const int buf = it & 1;
    const bool more = q + 1 < nq || c - 1 >= c_begin;
    if (q + 1 < nq) stage(c, q + 1, buf ^ 1);
    else if (c - 1 >= c_begin) stage(c - 1, 0, buf ^ 1);
    const bool landed = !misaligned && mbar_wait(&tbar[buf], (it >> 1) & 1);
    if (__syncthreads_or(!landed)) {
      // a tile did not arrive: report it, let the copy issued above drain, leave
      if (tid == 0) {
        report_timeout(&g_bwd2_status, a.status);
        if (!misaligned && more) mbar_wait(&tbar[buf ^ 1], ((it + 1) >> 1) & 1);
      }
      aborted = true;
      break;
    }
    const bool fw = q < nt - 1;
    const int jt = fw ? q : 2 * nt - 2 - q;  // tile within the chunk
    const int t0 = c * K + jt * KS;          // its first step
    const int steps = min(KS, min(c * K + K, g.T) - t0);
    const unsigned char* base = smem + (size_t)buf * L.tile;
    if (ST && a.conv_in && t0 < 3 && active && hf == 0) {
      T* xw = reinterpret_cast<T*>(smem + (size_t)buf * L.tile + L.x);
      const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * g.D + d;
      for (int r = 0; r < 3 - t0; ++r) xw[r * CH + ch] = ci[(size_t)(t0 + r) * g.D];
    }
    {
      const T* Bt = reinterpret_cast<const T*>(base + L.Bt);
      const T* Ct = reinterpret_cast<const T*>(base + L.Ct);
      // copy r, row j: position 8 h + 2 P + e holds state lane 8 h + 2 (P ^ r) + e
      for (int i = tid; i < KS * N; i += 128) {
        const float bv = Act<T>::ld(Bt + i), cv = fw ? 0.f : Act<T>::ld(Ct + i);
        const int j = i / N, n = i % N;
#pragma unroll
        for (int r = 0; r < NROT; ++r) {
          const int o = r * rot_stride(KT, N) + j * N + (n & ~7) + 2 * (((n >> 1) & 3) ^ r) + (n & 1);
          fB[o] = bv;
          if (!fw) fC[o] = cv;
        }
      }
    }
    __syncthreads();
    const T* xt = reinterpret_cast<const T*>(base + L.x);  // row r is step t0 - 3 + r
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const T* dgt = reinterpret_cast<const T*>(base + L.dg);
    const float* ckt = reinterpret_cast<const float*>(base + L.ck);
    float4* s0 = reinterpret_cast<float4*>(smem + L.scal) + ch;  // shared by the channel's threads, stride CH
    float4* s1 = s0 + (size_t)KT * CH;
    const size_t row0 = ((size_t)b * g.T + (size_t)t0) * g.D + d;

    if (fw) {
      // ---- forward item: this thread's lanes of the states through tile
      // jt, from the start state in this buffer (the chunk's checkpoint for
      // tile 0, else left by the forward item before) ----
      float2 hs[4];
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const int n = lane_of(P);
        hs[P] = make_float2(ckt[n * CH + ch], ckt[(n + 1) * CH + ch]);
      }
      for (int j = hf; j < steps; j += G) {
        const float xm3 = Act<T>::ld(xt + j * CH + ch);
        const float xm2 = Act<T>::ld(xt + (j + 1) * CH + ch);
        const float xm1 = Act<T>::ld(xt + (j + 2) * CH + ch);
        const float xv = Act<T>::ld(xt + (j + 3) * CH + ch);
        const float cpre = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
        const float u = cpre * sigmoid_f(cpre);
        const float delta = softplus_f(Act<T>::ld(drt + j * CH + ch) + dtb);
        *reinterpret_cast<float2*>(s0 + j * CH) = make_float2(delta, delta * u);
      }
      __syncwarp();
#pragma unroll 2
      for (int j = 0; j < steps; ++j) {
        const float2 v0 = *reinterpret_cast<const float2*>(s0 + j * CH);
        const float2 dl2 = f2b(v0.x);
        const float2 du2 = f2b(v0.y);
#pragma unroll
        for (int P = 0; P < 4; ++P) {
          const float2 bb = *reinterpret_cast<const float2*>(fBr + j * N + 2 * P);
          hs[P] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2[P])), hs[P], __fmul2_rn(du2, bb));
        }
      }
      if (jt + 1 < nt - 1) {
        // the state before tile jt + 1: a sub-checkpoint, read back by the
        // backward item of that tile with a tile copy
        float* skp = a.sk + ((size_t)slot * g.nsk + jt) * N * CH + ch;
        const uint64_t keep_policy = l2_evict_last_policy();
#pragma unroll
        for (int P = 0; P < 4; ++P) {
          const int n = lane_of(P);
          st_keep(skp + n * CH, hs[P].x, keep_policy);
          st_keep(skp + (n + 1) * CH, hs[P].y, keep_policy);
        }
        fence_proxy_async_global();
      }
      {
        // and the start state of the next item (the next forward item, or
        // the backward item of the last tile), whose copies bring none
        float* ckn = reinterpret_cast<float*>(smem + (size_t)(buf ^ 1) * L.tile + L.ck);
#pragma unroll
        for (int P = 0; P < 4; ++P) {
          const int n = lane_of(P);
          ckn[n * CH + ch] = hs[P].x;
          ckn[(n + 1) * CH + ch] = hs[P].y;
        }
      }
      __syncthreads();
      continue;
    }

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
          const float2 bb = *reinterpret_cast<const float2*>(fBr + j * N + 2 * P);
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
          const float2 bb = *reinterpret_cast<const float2*>(fBr + j * N + 2 * P);
          const float2 cc = *reinterpret_cast<const float2*>(fCr + j * N + 2 * P);
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
      const int t = t0 + j;
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
        const int t = t0 + j;
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
        dcs[KS * CH + ch] = v0;
        dcs[(KS + 1) * CH + ch] = v1;
        dcs[(KS + 2) * CH + ch] = v2;
      }
    }

    __syncthreads();
    if constexpr (DET) {  // this block's share, summed in a fixed order by m3_dbc_sum_kernel
      for (int i = tid; i < steps * 2 * N; i += 128) {
        const int j = i / (2 * N), l = i % (2 * N);
        float v = 0.f;
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) v += red[(j * 4 + ww) * 2 * N + l];
        a.dbc_part[(((size_t)b * g.T + t0 + j) * a.nblk + blockIdx.x) * 2 * N + l] = v;
      }
    } else {
      for (int i = tid; i < steps * 2 * N; i += 128) {
        const int j = i / (2 * N), l = i % (2 * N);
        float v = 0.f;
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) v += red[(j * 4 + ww) * 2 * N + l];
        float* dst = (l < N ? a.dB : a.dC) + ((size_t)b * g.T + t0 + j) * g.lddbc + (l & (N - 1));
        atomicAdd(dst, v);
      }
    }
    __syncthreads();
   }
  }

  if (!aborted) {
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
        // dc of steps 0, 1, 2 (zero past the sequence), kept in rows KS .. KS+2
        const float f0 = dcs[KS * CH + ch], f1 = dcs[(KS + 1) * CH + ch], f2 = dcs[(KS + 2) * CH + ch];
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
    if (!DET && a.fin) {
      // this block's sums, staged in the outputs' layout (d_a_log [CH][N],
      // d_conv_w [CH][4], then dD, d_dt_bias, d_conv_b [CH] each) in its tile
      // buffers, idle now, for the cluster's sum over the segments below
      float* sA = reinterpret_cast<float*>(smem);
      float* sW = sA + CH * N;
      float* sV = sW + CH * WC;
  #pragma unroll
      for (int P = 0; P < 4; ++P) {
        const int n = lane_of(P);  // dL/da_log = dL/dA * A, A = (A log2 e) ln 2
        sA[ch * N + n] = dAp[P].x * (a2[P].x * LN2);
        sA[ch * N + n + 1] = dAp[P].y * (a2[P].y * LN2);
      }
      if (hf == 0) {
  #pragma unroll
        for (int k = 0; k < WC; ++k) sW[ch * WC + k] = dcw[k];
        sV[ch] = dD_acc;
        sV[CH + ch] = ddtb_acc;
        sV[2 * CH + ch] = dcb_acc;
      }
    } else if (active) {
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
  }
  if constexpr (!DET) {
    if (a.fin) {
      // The S segments of this (channel block, batch) are one cluster; every
      // block passes both cluster barriers, aborted or not.
      cluster_sync_all();
      if (!aborted) {
        if constexpr (!SCAN) {
          // d_x at the last three steps of this segment: its own partial rows
          // plus the conv-input gradient of the next segment's first three
          // steps, written by the next block before the barrier
          if (s + 1 < g.S) {
            for (int i = tid; i < 3 * CH; i += 128) {
              const int j = i / CH, dd = d0 + i % CH;
              if (dd >= g.D) continue;
              const int t = t_end - 3 + j;
              float v = __ldcg(a.dxpart + (((size_t)b * g.S + s) * 3 + j) * g.D + dd);
  #pragma unroll
              for (int k = 0; k < WC; ++k) {
                const int tp = t + 3 - k;
                if (tp >= t_end && tp < g.T)
                  v = fmaf(__ldcg(a.dchead + (((size_t)b * g.S + s + 1) * 3 + (tp - t_end)) * g.D + dd),
                           a.conv_w[(size_t)dd * WC + k], v);
              }
              Act<T>::st(static_cast<T*>(a.dx) + ((size_t)b * g.T + t) * g.D + dd, v);
            }
          }
        }
        // parameter sums: four consecutive staged values per thread, summed
        // over the cluster's blocks in segment order, then added to the
        // outputs (one float4 atomic where the four are in range and 16-byte
        // aligned); block s takes every S-th group of 128 quads
        constexpr int U = CH * (N + 7) / 4;
        const int nch = min(CH, g.D - d0);
        const uint32_t sbase = smem_u32(smem);
        for (int u = s * 128 + tid; u < U; u += g.S * 128) {
          float4 v = ld_cluster_f4(cluster_addr(sbase + 16u * u, 0));
          for (int r = 1; r < g.S; ++r) {
            const float4 w4 = ld_cluster_f4(cluster_addr(sbase + 16u * u, r));
            v.x += w4.x;
            v.y += w4.y;
            v.z += w4.z;
            v.w += w4.w;
          }
          const int i = 4 * u;
          float* dst;
          int idx, lim;
          if (i < CH * N) {
            dst = a.d_a_log + (size_t)d0 * N;
            idx = i;
            lim = nch * N;
          } else if (i < CH * (N + WC)) {
            if (SCAN) continue;
            dst = a.d_conv_w + (size_t)d0 * WC;
            idx = i - CH * N;
            lim = nch * WC;
          } else {
            const int jv = i - CH * (N + WC), q = jv / CH;
            if (SCAN && q == 2) continue;
            dst = (q == 0 ? a.dD : q == 1 ? a.d_dt_bias : a.d_conv_b) + d0;
            idx = jv - q * CH;
            lim = nch;
          }
          if (idx + 4 <= lim && (reinterpret_cast<uintptr_t>(dst + idx) & 15u) == 0) {
            atomicAdd(reinterpret_cast<float4*>(dst + idx), v);
          } else {
            const float e4[4] = {v.x, v.y, v.z, v.w};
  #pragma unroll
            for (int e = 0; e < 4; ++e)
              if (idx + e < lim) atomicAdd(dst + idx + e, e4[e]);
          }
        }
      }
      cluster_sync_relaxed();  // no block leaves while the others may read its staging
    }
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_slot, a.tcols);
}


// the split kernel for (deterministic dB/dC, stop at du, carried state, d_state)
template <typename T, bool ST, bool SCAN, bool DET>
void (*bwd2_for(int N))(BwdArgs) {
  return N == 16 ? m3_bwd2_kernel<T, ST, SCAN, 16, DET>
       : N == 32 ? m3_bwd2_kernel<T, ST, SCAN, 32, DET> : m3_bwd2_kernel<T, ST, SCAN, 64, DET>;
}
template <typename T, bool DET>
void (*bwd2_pick(bool scan, bool st, int N))(BwdArgs) {
  return scan ? (st ? bwd2_for<T, true, true, DET>(N) : bwd2_for<T, false, true, DET>(N))
              : (st ? bwd2_for<T, true, false, DET>(N) : bwd2_for<T, false, false, DET>(N));
}
template <typename T>
void (*bwd2_kernel_for(bool det, bool scan, bool st, int N))(BwdArgs) {
  return det ? bwd2_pick<T, true>(scan, st, N) : bwd2_pick<T, false>(scan, st, N);
}

template void (*bwd2_kernel_for<float>(bool, bool, bool, int))(BwdArgs);
template void (*bwd2_kernel_for<__nv_bfloat16>(bool, bool, bool, int))(BwdArgs);

}  // namespace m3

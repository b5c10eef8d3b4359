// m3_fwd.cu -- the forward kernels (one thread per channel, and the split
// kernels with d_state / 8 threads per channel) and their launch.
#include "m3_common.cuh"

namespace m3 {

// nonzero once a kernel here gave up waiting for a tile copy
__device__ unsigned int g_fwd_status;

cudaError_t take_fwd_status(unsigned* out) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(v));
  if (e == cudaSuccess && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

// Wait for the tiles of staging buffer buf (its (it >> 1)-th use).  On a
// timeout every thread of the block learns it at the block barrier; thread
// 0 reports it and lets the copy it issued into the other buffer (if any)
// drain, and the caller leaves.  Returns false then.
__device__ __forceinline__ bool fwd_tiles_landed(uint64_t* tbar, int it, bool misaligned, bool other_in_flight,
                                                 unsigned* ws_status) {
  const int buf = it & 1;
  const bool landed = !misaligned && mbar_wait(&tbar[buf], (it >> 1) & 1);
  if (!__syncthreads_or(!landed)) return true;
  if (threadIdx.x == 0) {
    report_timeout(&g_fwd_status, ws_status);
    if (!misaligned && other_in_flight) mbar_wait(&tbar[buf ^ 1], ((it + 1) >> 1) & 1);
  }
  return false;
}

// ---------------------------------------------------------------------------
// forward: FINAL = run each segment from its true start state, write gated
// (+y) and a checkpoint every K steps; !FINAL = local pass from zero over
// segments 0..S-2 writing only the end state and the summed step size.
// Lanes are handled in pairs with packed f32x2 arithmetic.
// ---------------------------------------------------------------------------

template <typename T, bool FINAL>
__global__ void __launch_bounds__(GF) m3_fwd_kernel(const __grid_constant__ FwdArgs a) {
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
  float* fB = reinterpret_cast<float*>(smem + L.fB);
  float* fC = reinterpret_cast<float*>(smem + L.fC);

  // A tile's x, delta_raw, B (and z, C) rows arrive by tensor-map copies
  // issued by thread 0; rows past the sequence and channels past d_inner
  // arrive as zeros (rows past the segment are never read).
  __shared__ __align__(8) uint64_t tbar[2];  // tile copies into staging buffer 0 / 1
  if (tid == 0) {
    mbar_init(&tbar[0], 1);
    mbar_init(&tbar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  const bool misaligned = (smem_u32(smem) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  const uint32_t tile_bytes = (uint32_t)(((FINAL ? 3 : 2) * TT * GF + (FINAL ? 2 : 1) * TT * NS) * sizeof(T));
  auto stage = [&](int t0, int buf) {
    if (tid == 0 && !misaligned) {
      unsigned char* base = smem + (size_t)buf * L.tile;
      if (FINAL) bulk_wait_read();  // the output stores of the tile that last used this buffer
      fence_proxy_async();
      mbar_expect_tx(&tbar[buf], tile_bytes);
      tma_load_3d(base + L.x, &a.tm[TF_X], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.dr, &a.tm[TF_DR], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.Bt, &a.tm[TF_B], 0, t0, b, &tbar[buf]);
      if (FINAL) {
        tma_load_3d(base + L.z, &a.tm[TF_Z], d0, t0, b, &tbar[buf]);
        tma_load_3d(base + L.Ct, &a.tm[TF_C], 0, t0, b, &tbar[buf]);
      }
    }
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
    chain_segments<NS / 2, 1>(h, a2, a.agg_s, a.agg_h, NS, (size_t)b * g.S, 0, 1, s, g.D, d, active,
                              [](int i) { return 2 * i; });
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
  const bool want_y = a.y_dbg != nullptr;
  // checkpoints: the state before every step t with t % K == 0; kc = steps
  // from the current sub-tile's start to the next one, ck = that checkpoint
  // (running counters: no division per step or sub-tile)
  int kc = 0;
  float* ck = a.ckpt + (((size_t)b * g.nc + c_begin) * NS) * g.D + d;
  const size_t ck_step = (size_t)NS * g.D;
  // The final pass writes gated (and y) of a tile into the staging regions of
  // z (and delta_raw), which its scalar pass has consumed, and stores each
  // whole 8-step sub-tile with a tile copy; a sub-tile cut short by the end
  // of the segment (chunks under 8 steps) is written by the threads.
  for (int t0 = t_begin, it = 0; t0 < t_end; t0 += TT, ++it) {
    const int buf = it & 1;
    const bool more = t0 + TT < t_end;
    // the local pass issues the next tile's copies now; the final pass after
    // its first scalar sub-pass, when the stores that read that buffer are done
    if (!FINAL && more) stage(t0 + TT, buf ^ 1);
    if (!fwd_tiles_landed(tbar, it, misaligned, !FINAL && more, a.status)) return;
    unsigned char* base = smem + (size_t)buf * L.tile;
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
    T* og = reinterpret_cast<T*>(base + L.z);   // gated over z
    T* oy = reinterpret_cast<T*>(base + L.dr);  // y over delta_raw
    const int steps = min(TT, t_end - t0);
    for (int j0 = 0; j0 < steps; j0 += SUB) {
      const int ns = min(SUB, steps - j0);
      // scalar pass: independent per step (conv, SiLU, softplus, gate factor)
#pragma unroll
      for (int j = 0; j < SUB; ++j) {
        if (j >= ns) break;
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
      if (FINAL && j0 == 0 && more) stage(t0 + TT, buf ^ 1);
      // state pass: the only loop-carried dependence is h; a checkpoint at
      // every step jc = kc, kc + K, ... of this sub-tile
      const int tsub = t0 + j0;
      int jc = kc;
      const bool whole = tsub + SUB <= t_end;  // stored by a tile copy
#pragma unroll
      for (int j = 0; j < SUB; ++j) {
        if (j >= ns) break;
        if (FINAL && j == jc) {
          jc += g.K;
          if (active) {
#pragma unroll
            for (int i = 0; i < NS / 2; ++i) {
              ck[(size_t)(2 * i) * g.D] = h[i].x;
              ck[(size_t)(2 * i + 1) * g.D] = h[i].y;
            }
          }
          ck += ck_step;
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
          if (whole) {
            Act<T>::st(og + (j0 + j) * GF + tid, y * v.w);
            if (want_y) Act<T>::st(oy + (j0 + j) * GF + tid, y);
          } else if (active) {
            const size_t i = ((size_t)b * g.T + tsub + j) * g.D + d;
            Act<T>::st(static_cast<T*>(a.gated) + i, y * v.w);
            if (want_y) Act<T>::st(static_cast<T*>(a.y_dbg) + i, y);
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
      kc = jc - ns;  // the next checkpoint, from the next sub-tile's start
    }
    if (FINAL) {
      fence_proxy_async();  // this thread's output rows, before the tile stores read them
      __syncthreads();
      if (tid == 0) {
        // rows past the sequence and channels past d_inner are not written
        for (int j0 = 0; j0 < steps; j0 += SUB) {
          if (t0 + j0 + SUB > t_end) break;
          tma_store_3d(&a.tm[TF_OG], og + j0 * GF, d0, t0 + j0, b);
          if (want_y) tma_store_3d(&a.tm[TF_OY], oy + j0 * GF, d0, t0 + j0, b);
        }
        bulk_commit();
      }
    } else {
      __syncthreads();
    }
  }
  if (FINAL && tid == 0) bulk_wait_all();  // the tile stores are done before the block's memory goes
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
__global__ void __launch_bounds__(128) m3_fwd2_kernel(const __grid_constant__ FwdArgs a) {
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

  // x arrives with the three steps before the tile (row r = step t0 - 3 + r);
  // tiles come by tensor-map copies issued by thread 0, zeros outside the
  // tensor (rows past the segment are never read)
  __shared__ __align__(8) uint64_t tbar[2];  // tile copies into staging buffer 0 / 1
  if (tid == 0) {
    mbar_init(&tbar[0], 1);
    mbar_init(&tbar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  const bool misaligned = (smem_u32(smem) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  const uint32_t tile_bytes =
      (uint32_t)((((FINAL ? 3 : 2) * TT2 + 3) * CH + (FINAL ? 2 : 1) * TT2 * N) * sizeof(T));
  auto stage = [&](int t0, int buf) {
    if (tid == 0 && !misaligned) {
      unsigned char* base = smem + (size_t)buf * L.tile;
      fence_proxy_async();
      mbar_expect_tx(&tbar[buf], tile_bytes);
      tma_load_3d(base + L.x, &a.tm[TF_X], d0, t0 - 3, b, &tbar[buf]);
      tma_load_3d(base + L.dr, &a.tm[TF_DR], d0, t0, b, &tbar[buf]);
      tma_load_3d(base + L.Bt, &a.tm[TF_B], 0, t0, b, &tbar[buf]);
      if (FINAL) {
        tma_load_3d(base + L.z, &a.tm[TF_Z], d0, t0, b, &tbar[buf]);
        tma_load_3d(base + L.Ct, &a.tm[TF_C], 0, t0, b, &tbar[buf]);
      }
    }
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
    chain_segments<4, 2>(h, a2, a.agg_s, a.agg_h, N, (size_t)b * g.S, 0, 1, s, g.D, d, active,
                         [hf](int P) { return 8 * hf + 2 * P; });
  }
  float sdelta = 0.f;
  float4* scs = reinterpret_cast<float4*>(smem + L.sc) + ch;  // shared by the channel's threads, stride CH
  int kc = 0;  // steps left until the next checkpoint
  // the next checkpoint's lanes of this thread (a running pointer: no division)
  float* ck = a.ckpt + (((size_t)b * g.nc + c_begin) * N + 8 * hf) * g.D + d;
  const size_t ck_step = (size_t)N * g.D;
  for (int t0 = t_begin, it = 0; t0 < t_end; t0 += TT2, ++it) {
    const int buf = it & 1;
    if (t0 + TT2 < t_end) stage(t0 + TT2, buf ^ 1);
    if (!fwd_tiles_landed(tbar, it, misaligned, t0 + TT2 < t_end, a.status)) return;
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
      for (int i = tid; i < TT2 * N; i += 128) {
        fB[i] = Act<T>::ld(Bt + i);
        if (FINAL) fC[i] = Act<T>::ld(Ct + i);
      }
    }
    __syncthreads();
    const T* xt = reinterpret_cast<const T*>(base + L.x);
    const T* drt = reinterpret_cast<const T*>(base + L.dr);
    const T* zt = reinterpret_cast<const T*>(base + L.z);
    const int steps = min(TT2, t_end - t0);
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
            if (active) {
#pragma unroll
              for (int P = 0; P < 4; ++P) {
                ck[(size_t)(2 * P) * g.D] = h[P].x;
                ck[(size_t)(2 * P + 1) * g.D] = h[P].y;
              }
            }
            ck += ck_step;
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

// Tensor maps of the forward's tiles: boxes of ch channels x tt rows (x:
// tt + halo rows) and N x tt for B and C; tt is the kernel's staging tile.
template <typename T>
bool encode_fwd_maps(const Plan& p, int ch, int halo, int tt, FwdArgs& a) {
  const uint64_t es = sizeof(T), D = p.D, T_ = p.T, B = p.B, N = p.N, ld = p.ldbc;
  const uint32_t c = (uint32_t)ch, n = (uint32_t)p.N;
  const uint64_t adim[3] = {D, T_, B}, astr[2] = {D * es, T_ * D * es};
  const uint64_t bdim[3] = {N, T_, B}, bstr[2] = {ld * es, T_ * ld * es};
  const uint32_t rows = (uint32_t)tt;
  const uint32_t box_x[3] = {c, rows + halo, 1}, box_a[3] = {c, rows, 1}, box_b[3] = {n, rows, 1};
  const uint32_t box_o[3] = {c, SUB, 1};
  bool ok = encode_tile_map(&a.tm[TF_X], (int)es, 3, a.x, adim, astr, box_x) &&
            encode_tile_map(&a.tm[TF_DR], (int)es, 3, a.dr, adim, astr, box_a) &&
            encode_tile_map(&a.tm[TF_Z], (int)es, 3, a.z, adim, astr, box_a) &&
            encode_tile_map(&a.tm[TF_B], (int)es, 3, a.Bm, bdim, bstr, box_b) &&
            encode_tile_map(&a.tm[TF_C], (int)es, 3, a.Cm, bdim, bstr, box_b);
  if (ok && halo == 0) {  // the one-thread final pass stores its output sub-tiles
    ok = encode_tile_map(&a.tm[TF_OG], (int)es, 3, a.gated, adim, astr, box_o) &&
         (!a.y_dbg || encode_tile_map(&a.tm[TF_OY], (int)es, 3, a.y_dbg, adim, astr, box_o));
  }
  if (!ok) note(cudaErrorInvalidValue);
  return ok;
}

template <typename T>
m3_status launch_fwd(const Plan& p, FwdArgs a, cudaStream_t st) {
  const int groups = (p.D + GF - 1) / GF;
  const size_t smem = fwd_smem(sizeof(T)).total;
  a.g = Geo{p.B, p.T, p.D, p.K, p.nc, p.Sf, p.mf, p.ldbc, p.lddbc, p.KS, 0};
  cudaError_t e = cudaSuccess;
  if (p.fwd_tpc != 1) {  // split kernels, N / 8 threads per channel
    const int ch = 128 / (p.N / 8);
    const dim3 ga((p.D + ch - 1) / ch, p.Sf - 1, p.B), gf((p.D + ch - 1) / ch, p.Sf, p.B);
    const size_t smem2 = fwd2_smem(sizeof(T), p.N).total;
    if (!encode_fwd_maps<T>(p, ch, 3, TT2, a)) return M3_ERR_CUDA;
    void (*agg)(FwdArgs) = p.N == 16 ? m3_fwd2_kernel<T, false, 16>
                         : p.N == 32 ? m3_fwd2_kernel<T, false, 32> : m3_fwd2_kernel<T, false, 64>;
    void (*fin)(FwdArgs) = p.N == 16 ? m3_fwd2_kernel<T, true, 16>
                         : p.N == 32 ? m3_fwd2_kernel<T, true, 32> : m3_fwd2_kernel<T, true, 64>;
    if (p.Sf > 1) e = launch_k(agg, ga, 128, smem2, st, false, a);
    if (e == cudaSuccess) e = launch_k(fin, gf, 128, smem2, st, p.Sf > 1, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
  }
  if (!encode_fwd_maps<T>(p, GF, 0, TT, a)) return M3_ERR_CUDA;
  if (p.Sf > 1) e = launch_k(m3_fwd_kernel<T, false>, dim3(groups, p.Sf - 1, p.B), GF, smem, st, false, a);
  if (e == cudaSuccess)
    e = launch_k(m3_fwd_kernel<T, true>, dim3(groups, p.Sf, p.B), GF, smem, st, p.Sf > 1, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

template <typename T>
cudaError_t set_fwd_attrs() {
  const int es = sizeof(T);
  cudaError_t e;
  e = cudaFuncSetAttribute(m3_fwd_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)fwd_smem(es).total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_fwd_kernel<T, true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_fwd_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)fwd_smem(es).total);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_fwd_kernel<T, false>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
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
  return e;
}

template <typename T>
cudaError_t fwd_occupancy(int* blocks) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, m3_fwd_kernel<T, true>, GF,
                                                       fwd_smem(sizeof(T)).total);
}

template m3_status launch_fwd<float>(const Plan&, FwdArgs, cudaStream_t);
template m3_status launch_fwd<__nv_bfloat16>(const Plan&, FwdArgs, cudaStream_t);
template cudaError_t set_fwd_attrs<float>();
template cudaError_t set_fwd_attrs<__nv_bfloat16>();
template cudaError_t fwd_occupancy<float>(int*);
template cudaError_t fwd_occupancy<__nv_bfloat16>(int*);

}  // namespace m3

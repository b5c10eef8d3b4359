// m3_aux.cu -- the conv backward of the two-phase backward and the decode
// kernels, and their launch.
#include "m3_common.cuh"

namespace m3 {

// nonzero once a kernel here gave up waiting for a tile copy
__device__ unsigned int g_aux_status;

cudaError_t take_aux_status(unsigned* out) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_aux_status, sizeof(v));
  if (e == cudaSuccess && v) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_aux_status, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

template <typename T>
__global__ void __launch_bounds__(128) m3_conv_bwd_kernel(const __grid_constant__ ConvArgs a) {
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
  // the tile's rows arrive by tensor-map copies issued by thread 0 (zeros
  // outside [0, T) and past d_inner)
  __shared__ __align__(8) uint64_t tbar;
  const bool misaligned = (smem_u32(smem) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  if (tid == 0) {
    mbar_init(&tbar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0 && !misaligned) {
    const uint32_t bytes = (uint32_t)(((CT + 6) + (a.du_extra ? 2 : 1) * (CT + 3)) * 128 * sizeof(T));
    mbar_expect_tx(&tbar, bytes);
    tma_load_3d(xs, &a.tm[0], d0, t0 - 3, b, &tbar);
    tma_load_3d(us, &a.tm[1], d0, t0, b, &tbar);
    if (a.du_extra) tma_load_3d(es, &a.tm[2], d0, t0, b, &tbar);
  }
  const bool active = d < a.D;
  float w[WC] = {0.f, 0.f, 0.f, 0.f};
  float cb = 0.f;
  if (active) {
#pragma unroll
    for (int k = 0; k < WC; ++k) w[k] = a.conv_w[(size_t)d * WC + k];
    cb = a.conv_b[d];
  }
  const bool landed = !misaligned && mbar_wait(&tbar, 0);
  if (__syncthreads_or(!landed)) {
    if (tid == 0) report_timeout(&g_aux_status, a.status);
    return;
  }
  if (!active) return;  // no barriers below
  if (a.conv_in && t0 < 3) {
    // halo rows before step 0 (staged as zeros): the carried conv inputs
    const T* ci = static_cast<const T*>(a.conv_in) + (size_t)b * 3 * D + d;
    for (int r = 0; r < 3 - t0; ++r) xs[r * 128 + tid] = ci[(size_t)(t0 + r) * D];
  }
  // A tile whose steps and three look-ahead steps all lie inside the
  // sequence (every tile but the last one or two) runs without bounds checks.
  auto run = [&](auto full_tag) {
    constexpr bool FULL = decltype(full_tag)::value;
    // dc of steps t0 .. t1 + 2 (zero from step T on), then d_x of the tile
    float dcs[CT + 3];
    float dcb = 0.f, dcw[WC] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < CT + 3; ++j) {
      const int t = t0 + j;
      float dc = 0.f;
      if (FULL || t < a.T) {
        const float xm3 = Act<T>::ld(xs + j * 128 + tid);
        const float xm2 = Act<T>::ld(xs + (j + 1) * 128 + tid);
        const float xm1 = Act<T>::ld(xs + (j + 2) * 128 + tid);
        const float xv = Act<T>::ld(xs + (j + 3) * 128 + tid);
        float gu = Act<T>::ld(us + j * 128 + tid);
        if (a.du_extra) gu += Act<T>::ld(es + j * 128 + tid);
        const float c = fmaf(w[0], xm3, fmaf(w[1], xm2, fmaf(w[2], xm1, fmaf(w[3], xv, cb))));
        const float sc = sigmoid_f(c);
        dc = gu * (sc * fmaf(c, 1.f - sc, 1.f));
        if (j < CT && (FULL || t < t1)) {
          dcb += dc;
          dcw[0] = fmaf(dc, xm3, dcw[0]);
          dcw[1] = fmaf(dc, xm2, dcw[1]);
          dcw[2] = fmaf(dc, xm1, dcw[2]);
          dcw[3] = fmaf(dc, xv, dcw[3]);
        }
      }
      dcs[j] = dc;
    }
    T* const dxp = static_cast<T*>(a.dx) + ((size_t)b * a.T + t0) * D + d;
#pragma unroll
    for (int j = 0; j < CT; ++j) {
      const int t = t0 + j;
      if (FULL || t < t1) {
        float v = fmaf(dcs[j], w[3], fmaf(dcs[j + 1], w[2], fmaf(dcs[j + 2], w[1], dcs[j + 3] * w[0])));
        if (!FULL && a.g_conv && t >= a.T - 3)  // x[t] is also a conv-state output
          v += Act<T>::ld(static_cast<const T*>(a.g_conv) + ((size_t)b * 3 + t - (a.T - 3)) * D + d);
        Act<T>::st(dxp + (size_t)j * D, v);
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
  };
  if (t0 + CT + 3 <= a.T)
    run(std::true_type{});
  else
    run(std::false_type{});
}

// d_conv_b and d_conv_w from the per-(batch, tile) partials, summed in a
// fixed order (32 outputs per block, rows split over 16 warps, so enough
// loads are in flight to keep this short kernel off the latency floor).
__global__ void m3_conv_fin_kernel(ConvArgs a) {
  grid_dep_wait();  // the conv backward's partials
  __shared__ float part[16][33];
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
    for (; r + 16 < rows; r += 32) {
      v0 += P[(size_t)r * stride];
      v1 += P[(size_t)(r + 16) * stride];
    }
    if (r < rows) v0 += P[(size_t)r * stride];
    v0 += v1;
  }
  part[ry][cx] = v0;
  __syncthreads();
  if (ry != 0 || !ok) return;
  float v = 0.f;
#pragma unroll
  for (int k = 0; k < 16; k += 4)
    v += (part[k][cx] + part[k + 1][cx]) + (part[k + 2][cx] + part[k + 3][cx]);
  float* dst = j == 0 ? a.d_conv_b + d : a.d_conv_w + (size_t)d * WC + (j - 1);
  *dst = a.accumulate ? *dst + v : v;
}

// Each channel's N lanes are split over G = N / 16 neighbouring threads of
// a warp (16 lanes each; y is summed over the G threads with shuffles), so
// every d_state keeps 16 state lanes per thread.  R batch rows per thread
// (two when the grid is large enough) keep more loads in flight.  Each step
// issues all of its global loads before its barrier; B and C of the next
// step are staged into the other half of a double buffer.
// TL: the block's carried states arrive by one tensor-map copy into shared
// memory (hs[R][N][CH]), issued before the other loads and waited for after
// them; otherwise each thread loads its own lanes.  HS (with TL): the states
// stay in that shared-memory tile, are updated there and leave by one tile
// store, so a thread holds none in registers and more blocks fit per SM.
template <typename T, int N, int R, bool TL, bool HS>
__global__ void __launch_bounds__(GD, HS ? 8 : 5)  // blocks per SM: HS 8 (64 registers), else 5
m3_decode_kernel(const __grid_constant__ DecArgs a) {
  static_assert(!HS || TL, "shared-memory states arrive by the tile copy");
  constexpr int G = N / 16;       // threads per channel
  constexpr int CH = GD / G;      // channels per block
  constexpr int NB = 2 * N * R;   // B and C values of one step
  __shared__ float sBC[2][R][2 * N];
  __shared__ float sA[8][GD][2];  // A log2(e) of this thread's lanes
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(8) uint64_t tbar;
  const int tid = threadIdx.x;
  const bool misaligned = TL && (smem_u32(dsm) & 127u) != 0;  // tile copies need 128-byte aligned buffers
  if constexpr (TL) {
    if (tid == 0) {
      mbar_init(&tbar, 1);
      mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0 && !misaligned) {
      mbar_expect_tx(&tbar, (uint32_t)(R * N * CH * 4));
      tma_load_3d(dsm, &a.tm_h, blockIdx.x * CH, 0, blockIdx.y * R, &tbar);
    }
  }
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
    if constexpr (!TL) {
      const float* hp = a.h + ((size_t)rb[r] * N + 16 * q) * D + d;
#pragma unroll
      for (int i = 0; i < 8; ++i) h[r][i] = make_float2(hp[(size_t)(2 * i) * D], hp[(size_t)(2 * i + 1) * D]);
    }
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
  if constexpr (TL) {
    const bool landed = !misaligned && mbar_wait(&tbar, 0);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) report_timeout(&g_aux_status, nullptr);  // decode has no workspace
      return;
    }
    if constexpr (!HS) {
      const float* hs = reinterpret_cast<const float*>(dsm) + tid / G;
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          h[r][i] = make_float2(hs[((size_t)r * N + 16 * q + 2 * i) * CH], hs[((size_t)r * N + 16 * q + 2 * i + 1) * CH]);
      }
    }
  }
  // this thread's lane 16 q + 2 i (+1) of row r in the shared-memory tile
  float* const hsm = reinterpret_cast<float*>(dsm) + (size_t)16 * q * CH + tid / G;
  auto hs_at = [&](int r, int i) { return hsm + ((size_t)r * N + 2 * i) * CH; };

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
        if constexpr (HS) {
          float* hp = hs_at(r, k);
          const float2 hn = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2)), make_float2(hp[0], hp[CH]),
                                       __fmul2_rn(du2, bb));
          hp[0] = hn.x;
          hp[CH] = hn.y;
          y2 = __ffma2_rn(cc, hn, y2);
        } else {
          h[r][k] = __ffma2_rn(ex2x2(__fmul2_rn(dl2, a2)), h[r][k], __fmul2_rn(du2, bb));
          y2 = __ffma2_rn(cc, h[r][k], y2);
        }
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
  if constexpr (HS) {
    // the updated tile back by one tile store (lanes of channels past
    // d_inner and rows past the batch are not written); the block's shared
    // memory stays until the store has read it
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      tma_store_3d(&a.tm_h, dsm, blockIdx.x * CH, 0, blockIdx.y * R);
      bulk_commit();
      bulk_wait_read();
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!ron[r]) continue;
    if constexpr (!HS) {
      float* hp = a.h + ((size_t)rb[r] * N + 16 * q) * D + d;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        hp[(size_t)(2 * i) * D] = h[r][i].x;
        hp[(size_t)(2 * i + 1) * D] = h[r][i].y;
      }
    }
    if (q == 0) {
      T* cp = static_cast<T*>(a.conv) + (size_t)rb[r] * 3 * D + d;
      Act<T>::st(cp, xm3[r]);
      Act<T>::st(cp + D, xm2[r]);
      Act<T>::st(cp + 2 * D, xm1[r]);
    }
  }
}

template <typename T, int N, int R>
cudaError_t launch_decode_r(const DecArgs& a0, cudaStream_t st) {
  constexpr int CH = GD / (N / 16);
  const dim3 grid((unsigned)((a0.D + CH - 1) / CH), (unsigned)((a0.B + R - 1) / R));
  // the carried states in and out by tile copies, kept in shared memory in
  // between, when their layout allows a tile map (measured on GB300, 64
  // sequences of d_inner 5120: 8 % faster than per-thread loads into
  // registers for d_state 16, 19-23 % for 32 and 64)
  if (reinterpret_cast<uintptr_t>(a0.h) % 16 == 0 && a0.D % 4 == 0) {
    DecArgs a = a0;
    const uint64_t dim[3] = {(uint64_t)a.D, (uint64_t)N, (uint64_t)a.B};
    const uint64_t str[2] = {(uint64_t)a.D * 4, (uint64_t)N * a.D * 4};
    const uint32_t box[3] = {(uint32_t)CH, (uint32_t)N, (uint32_t)R};
    if (!encode_tile_map(&a.tm_h, 4, 3, a.h, dim, str, box)) return cudaErrorInvalidValue;
    m3_decode_kernel<T, N, R, true, true><<<grid, GD, (size_t)R * N * CH * 4, st>>>(a);
  } else {
    m3_decode_kernel<T, N, R, false, false><<<grid, GD, 0, st>>>(a0);
  }
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

template <typename T>
cudaError_t launch_conv_bwd(ConvArgs a, dim3 grid, cudaStream_t s) {
  const uint64_t es = sizeof(T), D = a.D, T_ = a.T, B = a.B;
  const uint64_t dim[3] = {D, T_, B}, str[2] = {D * es, T_ * D * es};
  const uint32_t box_x[3] = {128, CT + 6, 1}, box_u[3] = {128, CT + 3, 1};
  if (!encode_tile_map(&a.tm[0], (int)es, 3, a.x, dim, str, box_x) ||
      !encode_tile_map(&a.tm[1], (int)es, 3, a.du, dim, str, box_u) ||
      (a.du_extra && !encode_tile_map(&a.tm[2], (int)es, 3, a.du_extra, dim, str, box_u)))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_k(m3_conv_bwd_kernel<T>, grid, 128, conv_smem(sizeof(T)).total, s, false, a);
  if (e == cudaSuccess)
    e = launch_k(m3_conv_fin_kernel, dim3((unsigned)((5 * (size_t)a.D + 31) / 32)), 512, 0, s, true, a);
  return e;
}

template <typename T>
cudaError_t set_aux_attrs() {
  const int es = sizeof(T);
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(m3_conv_bwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)conv_smem(es).total);
  return e;
}

template cudaError_t launch_conv_bwd<float>(ConvArgs, dim3, cudaStream_t);
template cudaError_t launch_conv_bwd<__nv_bfloat16>(ConvArgs, dim3, cudaStream_t);
template cudaError_t launch_decode_n<float>(int, const DecArgs&, cudaStream_t, int);
template cudaError_t launch_decode_n<__nv_bfloat16>(int, const DecArgs&, cudaStream_t, int);
template cudaError_t set_aux_attrs<float>();
template cudaError_t set_aux_attrs<__nv_bfloat16>();

}  // namespace m3

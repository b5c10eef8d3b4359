// m3_api.cu -- the C ABI of the selective-scan layer core (include/m3scan.h):
// argument validation, the launch plan (chunk, time segments, workspace,
// kernel variants), per-device set-up, and the entry points.
//
// What is computed follows the mamba-rs pages: src/mamba_ssm/gpu/
// forward_mixed.rs (0.3.1), steps F4a conv1d + SiLU, F4c softplus, F4d the
// selective scan with the D skip, F4e gating, and the backward scratch list
// of the same page; A = -exp(a_log) from trainer.rs (0.7.3),
// recompute_a_neg_all.  The design is not the pages': they save the f32
// state before every step (h_saved, B*(T+1)*d_inner*d_state) and the
// discretisation da_exp per step.  Here the forward keeps a channel's state
// lanes in registers and writes only the state at the start of each chunk
// of K steps; the backward recomputes one chunk at a time into tensor memory
// and runs the reverse-time pass from there (m3_fwd.cu, m3_bwd.cu).
//
// Work decomposition.  A block owns (batch b, a group of channels, one time
// segment).  When batch x channel groups alone cannot fill the GPU, time is
// split into S segments of whole chunks.  The scan is linear in the state,
// so a segment's effect on the next is (decay, local end state): an
// aggregate pass computes it per segment and the main kernel chains the
// earlier segments' aggregates to its true start state.  The backward does
// the same in reverse time for the adjoint state.  dB and dC are sums over
// channels (warp shuffles, shared memory, one f32 global reduction per
// (t, n) per block).  Parameter gradients: the split main kernel over
// several segments adds each block's sums into the outputs with f32
// reductions; otherwise (and always when deterministic sums are asked for)
// they are per-(batch, segment) partials that a tail kernel sums in a fixed
// order.

#include <mutex>

#include "m3_common.cuh"

// Backward scratch owned by the library itself, for m3scan_bwd_noalloc.
// Every GPU that loads this library holds these bytes until the process
// exits.  Host code must not use the name as an address: it is fetched per
// device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[M3SCAN_NOALLOC_SCRATCH_BYTES];

namespace m3 {

// Identity of the calling thread's current CUDA context: 0 when there is
// none yet or the driver cannot say.  A context that was torn down and
// created again (cudaDeviceReset) gets a new identity, so the per-device
// caches below redo their set-up for it instead of reusing what belonged to
// the old one (function attributes, a symbol's device address).
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static const GetCurrentFn get_current = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<GetCurrentFn>(f);
  }();
  static const GetIdFn get_id = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<GetIdFn>(f);
  }();
  cudaGetLastError();  // a failed lookup leaves no error behind
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct DevInfo {
  bool attrs = false;
  unsigned long long ctx = 0;  // context the attributes were set in (0: unknown)
  int sms = 0;
  int smem_per_sm = 0;
  int occ_fwd[2][KT + 1];  // [dtype][backward tile] blocks per SM, 0 = not yet queried
  int occ_bwd[2][KT + 1];
};

std::mutex g_mu;
DevInfo g_dev[64];
thread_local cudaError_t g_last_cuda = cudaSuccess;  // last CUDA error this thread saw

// Record a failed CUDA call (and clear the runtime's sticky-free error state).
cudaError_t note(cudaError_t e) {
  if (e != cudaSuccess) {
    g_last_cuda = e;
    cudaGetLastError();
  }
  return e;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

bool encode_tile_map(CUtensorMap* map, int es, int rank, const void* ptr, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es1[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es1[i] = 1;
    if (i + 1 < rank) gs[i] = strides[i];
  }
  const CUresult r = fn(map, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs, bx, es1, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T>
cudaError_t set_attrs() {
  cudaError_t e = set_fwd_attrs<T>();
  if (e == cudaSuccess) e = set_bwd_attrs<T>();
  if (e == cudaSuccess) e = set_aux_attrs<T>();
  return e;
}

// Device facts for the current device: kernel attributes are set once per
// device (with that device current), occupancy is queried once per backward
// tile length (chunk = that tile, at most KT).
cudaError_t device_info(int chunk, int ai, int* sms, int* occ_f, int* occ_b, int* smem_sm = nullptr) {
  if (chunk < 1 || chunk > KT) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& di = g_dev[dev];
  const unsigned long long ctx = current_context_id();
  if (!di.attrs || (ctx != 0 && di.ctx != 0 && ctx != di.ctx)) {
    di.attrs = false;
    e = set_attrs<float>();
    if (e != cudaSuccess) return e;
    e = set_attrs<__nv_bfloat16>();
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    for (int a = 0; a < 2; ++a)
      for (int k = 0; k <= KT; ++k) di.occ_fwd[a][k] = di.occ_bwd[a][k] = 0;
    di.attrs = true;
    di.ctx = current_context_id();  // the set-up above made the context current if it was not
  }
  if (occ_f && di.occ_fwd[ai][chunk] == 0) {
    int of = 0, ob = 0;
    if (ai == 1) {
      e = fwd_occupancy<__nv_bfloat16>(&of);
      if (e == cudaSuccess) e = bwd_occupancy<__nv_bfloat16>(chunk, di.smem_per_sm, &ob);
    } else {
      e = fwd_occupancy<float>(&of);
      if (e == cudaSuccess) e = bwd_occupancy<float>(chunk, di.smem_per_sm, &ob);
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

// Backward segment count by wave fill: per_seg blocks per segment, W blocks
// resident at once.  Among splits with at least two chunks per segment and
// at most six waves of blocks, take the one whose last wave is fullest
// (blocks / (waves * W)), less 0.01 per wave.  Measured on GB300: the
// backward's time follows the filled fraction of its waves closely (a
// nearly empty last wave costs as much as a full one) and grows slowly with
// the number of segments.
int best_bwd_segments(int nc, int K, int64_t per_seg, int64_t W) {
  if (per_seg < 1) per_seg = 1;
  if (W < 1) W = 1;
  int64_t s_max = 6 * W / per_seg;
  // at least two chunks per segment, or one chunk once a chunk spans
  // several tiles (it is then long enough on its own)
  const int64_t min_chunks = K > KT ? 1 : 2;
  const int64_t cap = (nc + min_chunks - 1) / min_chunks;
  if (s_max > cap) s_max = cap;
  if (s_max > 65535) s_max = 65535;
  if (s_max < 1) s_max = 1;
  int best_S = 1;
  double best = -1.0;
  for (int64_t want = 1; want <= s_max; ++want) {
    int S = 1, m = 1;
    fix_segments(nc, K, (int)want, &S, &m);
    const int64_t n = per_seg * S;
    const int64_t waves = (n + W - 1) / W;
    const double score = (double)n / (double)(waves * W) - 0.01 * (double)waves;
    if (score > best + 1e-9) {
      best = score;
      best_S = S;
    }
  }
  return best_S;
}

// The checkpoint interval a call gets when it asks for none.  Measured on
// GB300 (bf16, long-sequence and Mamba-130M-like layers): 8-step chunks,
// whose backward recomputes each tile straight from its checkpoint, run
// fwd+bwd 16-19 % faster than 64- or 128-step chunks, whose backward first
// recomputes the sub-checkpoints of every chunk; the layer core is bound by
// instruction issue, not by the 16 bytes per element the 8-step checkpoints
// add to HBM traffic.
int default_chunk(int64_t seq_len) {
  (void)seq_len;
  return KSHORT;
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
  // a chunk longer than the backward's on-chip tile is a whole number of tiles
  if (dm->chunk > KT && dm->chunk % KT != 0) return M3_ERR_UNSUPPORTED;
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
  if (dm->deterministic != 0 && dm->deterministic != 1) return M3_ERR_DIMS;
  if (dm->reserved0 != 0) return M3_ERR_DIMS;
  return M3_OK;
}

m3_status make_plan(const m3_dims* dm, m3_dtype act, Plan* p) {
  m3_status st = validate_dims(dm, act);
  if (st != M3_OK) return st;
  p->B = (int)dm->batch;
  p->T = (int)dm->seq_len;
  p->D = (int)dm->d_inner;
  p->N = (int)dm->d_state;
  // default checkpoint interval
  p->K = dm->chunk ? (int)dm->chunk : default_chunk(dm->seq_len);
  p->nc = (p->T + p->K - 1) / p->K;
  p->KS = p->K < KT ? p->K : KT;
  {
    const int nt_max = (p->K + p->KS - 1) / p->KS;
    p->nsk = nt_max > 2 ? nt_max - 2 : 0;
  }
  p->ldbc = dm->bc_stride ? (int)dm->bc_stride : p->N;
  p->lddbc = dm->dbc_stride ? (int)dm->dbc_stride : p->N;
  const int groups_f = (p->D + GF - 1) / GF;
  const int groups_b = (p->D + GB - 1) / GB;
  int want_f = 1, want_b = 1;
  int64_t wave_b = 3 * 152;  // one-thread backward blocks resident at once
  int64_t wave_f = 6 * 152;  // one-thread forward blocks resident at once
  bool auto_split_b = false;  // backward kernel variant decided with its segments
  if (dm->segments > 0) {
    want_f = want_b = (int)dm->segments;
  } else if ((int64_t)p->B * p->T * p->D > 0) {
    int sms = 0, of = 0, ob = 0;
    if (note(device_info(KT, act == M3_BF16 ? 1 : 0, &sms, &of, &ob)) != cudaSuccess)
      return M3_ERR_CUDA;
    want_f = choose_segments(p->nc, p->K, (int64_t)p->B * groups_f, (int64_t)sms * of, 2);
    wave_b = (int64_t)sms * 3;  // three resident one-thread blocks per SM (measured; the
                                // occupancy query reports fewer)
    wave_f = (int64_t)sms * of;
    // backward: the one-thread kernels (three blocks per SM) unless even
    // their best split leaves the GPU less than one wave, then the split
    // kernels (four blocks per SM, 128 / (d_state / 8) channels per block)
    const int tpc = (int)dm->threads_per_channel;
    bool split = p->N != NS || tpc == 2;
    if (!split) {
      want_b = best_bwd_segments(p->nc, p->K, (int64_t)p->B * groups_b, wave_b);
      int Sb1 = 1, mb1 = 1;
      fix_segments(p->nc, p->K, want_b, &Sb1, &mb1);
      // (chunks of several tiles keep one thread per channel: the split
      // kernels' extra per-step work would be paid on every forward item too)
      split = tpc == 0 && p->K <= KT && (int64_t)p->B * groups_b * Sb1 <= wave_b;
      auto_split_b = split;
    }
    if (split) {
      const int ch = 128 / (p->N / 8);
      want_b = best_bwd_segments(p->nc, p->K, (int64_t)p->B * ((p->D + ch - 1) / ch), (int64_t)sms * 4);
    }
  }
  if (p->nc == 0) {
    p->Sf = p->Sb = 1;
    p->mf = p->mb = 0;
  } else {
    fix_segments(p->nc, p->K, want_f, &p->Sf, &p->mf);
    fix_segments(p->nc, p->K, want_b, &p->Sb, &p->mb);
  }
  const bool empty = (size_t)p->B * p->T * p->D == 0;
  // d_state 16: the split kernels (two threads per channel) when the
  // one-thread grid fills less than one wave (three backward, six forward
  // blocks per SM on a 152-SM GPU, or the device's figures when the
  // segments were chosen for it); wider states: always the split kernels,
  // d_state / 8 threads per channel
  p->fwd_tpc = p->bwd_tpc = dm->threads_per_channel;
  if (p->fwd_tpc == 0) p->fwd_tpc = (int64_t)p->B * groups_f * p->Sf <= wave_f ? 2 : 1;
  if (p->bwd_tpc == 0)
    p->bwd_tpc = (auto_split_b || (dm->segments > 0 && (int64_t)p->B * groups_b * p->Sb <= wave_b)) ? 2 : 1;
  if (p->N != NS) p->fwd_tpc = p->bwd_tpc = 2;
  if (p->fwd_tpc == 2) p->fwd_tpc = p->N / 8;
  if (p->bwd_tpc == 2) p->bwd_tpc = p->N / 8;
  const size_t B = p->B, D = p->D;
  const size_t N = p->N;
  p->ckpt_bytes = B * p->nc * N * D * 4;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  // forward section, after the status block
  off = STATUS_BYTES;
  p->f_aggh = p->f_aggs = 0;
  if (p->Sf > 1) {
    p->f_aggh = take(B * p->Sf * N * D * 4);
    p->f_aggs = take(B * p->Sf * D * 4);
  }
  size_t fwd_total = off;
  // backward section (reuses the same bytes)
  off = STATUS_BYTES;
  p->det = dm->deterministic != 0;
  p->fin = !p->det && p->bwd_tpc != 1 && p->Sb > 1 && p->Sb <= FIN_MAX;
  // per-(batch, segment) parameter partials, unless the main kernel adds
  // its sums into the outputs
  p->b_part = p->fin ? 0 : take(B * p->Sb * (N + 8) * D * 4);
  p->b_q = p->b_sd = p->b_dxpart = p->b_dchead = 0;
  if (p->Sb > 1) {
    p->b_q = take(B * p->Sb * N * D * 4);
    p->b_sd = take(B * p->Sb * D * 4);
    p->b_dxpart = take(B * p->Sb * 3 * D * 4);
    p->b_dchead = take(B * p->Sb * 3 * D * 4);
  }
  // deterministic dB/dC: one partial row of 2N floats per (batch, step,
  // channel block of the backward's main kernel)
  p->dblk = (p->D + (p->bwd_tpc != 1 ? 128 / p->bwd_tpc : GB) - 1) / (p->bwd_tpc != 1 ? 128 / p->bwd_tpc : GB);
  p->b_dbc = p->det ? take(B * (size_t)p->T * p->dblk * 2 * N * 4) : 0;
  // sub-checkpoints: the states before tiles 1 .. nt-2 of the chunk a block
  // of the main kernel is working on
  {
    const size_t ch = p->bwd_tpc != 1 ? 128 / p->bwd_tpc : GB;
    const size_t blocks = (size_t)p->dblk * p->Sb * B;
    p->b_sk = p->nsk > 0 && !empty ? take(blocks * p->nsk * N * ch * 4) : 0;
  }
  size_t bwd_total = off;
  // conv backward of the two-phase backward (its own call): CT-step tiles
  p->ctile = CT;
  p->cntiles = (p->T + CT - 1) / CT;
  off = STATUS_BYTES;
  p->c_part = take(B * (size_t)p->cntiles * 5 * D * 4);
  const size_t conv_total = off;
  if (conv_total > bwd_total) bwd_total = conv_total;
  p->ws_bytes = fwd_total > bwd_total ? fwd_total : bwd_total;
  if (p->ws_bytes < STATUS_BYTES) p->ws_bytes = STATUS_BYTES;
  p->fwd_launches = empty ? 0 : (p->Sf > 1 ? 2 : 1);
  p->bwd_launches = empty ? 0 : (p->Sb > 1 ? 2 : 1) + (p->fin ? 0 : 1) + (p->det ? 1 : 0);
  return M3_OK;
}

// The device must have this library's kernels registered: fail early and
// cleanly when the attribute setup cannot run (no device, wrong arch).
m3_status ensure_device(int chunk, int ai, int* smem_sm) {
  int of = 0, ob = 0;
  if (note(device_info(chunk, ai, nullptr, &of, &ob, smem_sm)) != cudaSuccess) return M3_ERR_CUDA;
  return M3_OK;
}

}  // namespace m3

using namespace m3;

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
    case M3_ERR_TIMEOUT:
      return "M3_ERR_TIMEOUT: a kernel gave up waiting for a tile copy; that call's outputs are incomplete";
  }
  return "unknown m3_status";
}

int32_t m3scan_version(void) { return 10100; }

m3_status m3scan_selftest_wait_timeout(void* workspace, m3_stream_t stream) {
  if (workspace && !aligned(workspace, 256)) return M3_ERR_ALIGN;
  if (note(launch_wait_timeout(static_cast<unsigned*>(workspace), reinterpret_cast<cudaStream_t>(stream))) !=
      cudaSuccess)
    return M3_ERR_CUDA;
  return M3_OK;
}

m3_status m3scan_get_status(const void* workspace, m3_stream_t stream, m3_status* device_status) {
  if (!workspace || !device_status) return M3_ERR_NULL;
  if (!aligned(workspace, 256)) return M3_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned word = 0;
  void* w = const_cast<void*>(workspace);
  if (note(cudaMemcpyAsync(&word, w, sizeof(word), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      note(cudaStreamSynchronize(s)) != cudaSuccess)
    return M3_ERR_CUDA;
  if (word != 0 && note(cudaMemsetAsync(w, 0, sizeof(word), s)) != cudaSuccess) return M3_ERR_CUDA;
  *device_status = word ? M3_ERR_TIMEOUT : M3_OK;
  return M3_OK;
}

m3_status m3scan_device_status(int32_t* out) {
  if (!out) return M3_ERR_NULL;
  unsigned vf = 0, vb = 0, v2 = 0, va = 0;
  if (note(take_fwd_status(&vf)) != cudaSuccess || note(take_bwd_status(&vb)) != cudaSuccess ||
      note(take_bwd2_status(&v2)) != cudaSuccess || note(take_aux_status(&va)) != cudaSuccess)
    return M3_ERR_CUDA;
  *out = (int32_t)(vf | vb | v2 | va);
  return M3_OK;
}

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
  // a workspace is needed over several time segments; one that is given
  // must be planned-size either way (its status block records failures)
  if (p.Sf > 1 && !workspace) return M3_ERR_WORKSPACE;
  if (workspace) {
    if (workspace_bytes < p.ws_bytes) return M3_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return M3_ERR_ALIGN;
  }
  int smem_sm = 0;
  if (ensure_device(KT, act == M3_BF16 ? 1 : 0, &smem_sm) != M3_OK) return M3_ERR_CUDA;
  FwdArgs a{};
  a.x = x; a.dr = delta_raw; a.z = z; a.Bm = Bm; a.Cm = Cm;
  a.conv_w = conv_w; a.conv_b = conv_b; a.dt_bias = dt_bias; a.a_log = a_log; a.Dp = D;
  a.gated = gated; a.y_dbg = y_dbg; a.ckpt = ckpt;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.agg_h = p.Sf > 1 ? reinterpret_cast<float*>(ws + p.f_aggh) : nullptr;
  a.agg_s = p.Sf > 1 ? reinterpret_cast<float*>(ws + p.f_aggs) : nullptr;
  a.h_in = sv.ssm_state; a.conv_in = sv.conv_state;
  a.h_out = sv.ssm_state_out; a.conv_out = sv.conv_state_out;
  a.status = static_cast<unsigned*>(workspace);
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
  if (ensure_device(KT, act == M3_BF16 ? 1 : 0, &smem_sm) != M3_OK) return M3_ERR_CUDA;
  BwdArgs a{};
  a.x = x; a.dr = delta_raw; a.z = z; a.Bm = Bm; a.Cm = Cm; a.dg = d_gated;
  a.conv_w = conv_w; a.conv_b = conv_b; a.dt_bias = dt_bias; a.a_log = a_log; a.Dp = D;
  a.ckpt = ckpt;
  a.dx = d_x; a.ddr = d_delta_raw; a.dz = dz; a.du_dbg = du_dbg;
  a.dB = dB; a.dC = dC;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.partials = reinterpret_cast<float*>(ws + p.b_part);
  a.dbc_part = p.det ? reinterpret_cast<float*>(ws + p.b_dbc) : nullptr;
  a.nblk = p.dblk;
  if (p.Sb > 1) {
    a.q = reinterpret_cast<float*>(ws + p.b_q);
    a.sd = reinterpret_cast<float*>(ws + p.b_sd);
    a.dxpart = reinterpret_cast<float*>(ws + p.b_dxpart);
    a.dchead = reinterpret_cast<float*>(ws + p.b_dchead);
  }
  a.fin = p.fin ? 1 : 0;
  // stopping at du leaves the conv parameters' grads alone
  a.d_conv_w = scan ? nullptr : d_conv_w; a.d_conv_b = scan ? nullptr : d_conv_b;
  a.d_dt_bias = d_dt_bias; a.d_a_log = d_a_log; a.dD = dD;
  a.accumulate = dims->accumulate_param_grads ? 1 : 0;
  a.conv_in = sv.conv_state; a.g_h = sv.d_ssm_state_out; a.g_conv = sv.d_conv_state_out;
  a.d_h_in = sv.d_ssm_state; a.d_conv_in = sv.d_conv_state;
  a.status = reinterpret_cast<unsigned*>(ws);
  a.sk = p.nsk > 0 ? reinterpret_cast<float*>(ws + p.b_sk) : nullptr;
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
  if (ensure_device(KT, act == M3_BF16 ? 1 : 0, &smem_sm) != M3_OK) return M3_ERR_CUDA;
  ConvArgs a{};
  a.B = p.B; a.T = p.T; a.D = p.D; a.tile = p.ctile; a.ntiles = p.cntiles;
  a.x = x; a.du = du; a.du_extra = du_extra; a.conv_w = conv_w; a.conv_b = conv_b; a.dx = d_x;
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + p.c_part);
  a.conv_in = sv.conv_state; a.g_conv = sv.d_conv_state_out; a.d_conv_in = sv.d_conv_state;
  a.d_conv_w = d_conv_w; a.d_conv_b = d_conv_b;
  a.accumulate = dims->accumulate_param_grads ? 1 : 0;
  a.status = static_cast<unsigned*>(workspace);
  const dim3 grid((unsigned)((p.D + 127) / 128), (unsigned)p.cntiles, (unsigned)p.B);
  cudaError_t e = act == M3_BF16 ? launch_conv_bwd<__nv_bfloat16>(a, grid, s) : launch_conv_bwd<float>(a, grid, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}


}  // extern "C"

namespace {

std::mutex g_noalloc_mu;
struct NoallocAddr {
  void* addr = nullptr;        // device address of g_noalloc_scratch
  unsigned long long ctx = 0;  // in this context (0: unknown)
};
NoallocAddr g_noalloc_addr[64];  // per device

// Set-up for m3scan_bwd_noalloc, once per device and context, with that
// device current: look up the device address of the library's scratch
// array.  A new context on the device (after cudaDeviceReset the module is
// loaded again and the array may sit elsewhere) looks it up again; when the
// driver cannot identify contexts it is looked up on every call.
m3_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return M3_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoallocAddr& na = g_noalloc_addr[dev];
  const unsigned long long ctx = current_context_id();
  if (!na.addr || ctx == 0 || ctx != na.ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      note(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      na.addr = nullptr;
      return M3_ERR_CUDA;
    }
    na.addr = p;
    na.ctx = current_context_id();  // the look-up made the context current if it was not
  }
  *out = na.addr;
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
  if (note(device_info(KT, act == M3_BF16 ? 1 : 0, &sms, &of, &ob)) != cudaSuccess)
    return M3_ERR_CUDA;
  const cudaError_t e = act == M3_BF16 ? launch_decode_n<__nv_bfloat16>(n, a, s, sms)
                                       : launch_decode_n<float>(n, a, s, sms);
  return note(e) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

}  // extern "C"

// Host side of the C ABI declared in include/qkvp.h: argument validation,
// tensor-map encoding, workspace layout and the launch sequence of each call.
// No call allocates device memory and none synchronises the host, except
// qkvp_poll_device_status.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "kernels.cuh"

using namespace qkvp;

namespace {

uint64_t g_timeout_ns = 2000000000ull;
// GEMMs run on CTA pairs (bit 0 forward, bit 1 dX, bit 2 dW).  The dX and
// dW GEMMs gain from pairs (their main loops are bound by shared-memory
// bandwidth, which pairs relieve); the forward GEMM, bound by its epilogue,
// does not.
int g_pair_mask = 6;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D map: `inner` elements per row (contiguous), `outer` rows, rows
// `row_bytes` apart.
bool map2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
           uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a [d2][d1][d0] row-major tensor.
bool map3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
           uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static std::atomic<int> cache[64];   // per device, written once (any thread may race to write the same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int qkvp::check_dims(const qkvp_dims* d) {
  if (!d) return QKVP_ERR_INVALID_ARGUMENT;
  if (d->T < 1 || d->D < 1 || d->H < 1 || d->d_qk < 1 || d->d_v < 1) return QKVP_ERR_INVALID_ARGUMENT;
  if (d->T > (1 << 24)) return QKVP_ERR_UNSUPPORTED;
  if (d->D % 128 != 0 || d->D > 16384) return QKVP_ERR_UNSUPPORTED;
  if (d->H > 128) return QKVP_ERR_UNSUPPORTED;
  if (d->d_qk != 64 && d->d_qk != 96 && d->d_qk != 128) return QKVP_ERR_UNSUPPORTED;
  if (d->d_v != 128) return QKVP_ERR_UNSUPPORTED;
  return QKVP_OK;
}

namespace {

// Workspace: [status 256 B][x amax partials][dY amax partials][dW partials]
// (and, for the packed projection, [dY row means])
constexpr size_t kStatusBytes = 256;
constexpr int kMaxParts = 4096;
constexpr size_t kPartsBytes = kMaxParts * sizeof(float);
constexpr int kMaxSplits = 16;

struct DwShape {
  int bn, m_tiles, n_tiles, kblocks_total;
};
// Tiles of a split-over-tokens weight gradient [R, C] from T tokens.
DwShape dw_shape_rc(int R, int C, int T) {
  DwShape s;
  s.bn = C % 256 == 0 ? 256 : 128;
  s.m_tiles = (R + 127) / 128;
  s.n_tiles = C / s.bn;
  s.kblocks_total = (T + 127) / 128;
  return s;
}
DwShape dw_shape(const qkvp_dims* d) { return dw_shape_rc(d->H * (2 * d->d_qk + d->d_v), d->D, d->T); }
size_t dw_partial_bytes(const DwShape& s, int splits) {
  return static_cast<size_t>(splits) * s.m_tiles * s.n_tiles * s.bn * 128 * sizeof(float);
}
size_t ws_bytes_for_shape(const DwShape& s) { return kStatusBytes + 2 * kPartsBytes + dw_partial_bytes(s, kMaxSplits); }
// The packed projection's workspace also holds the dY passes' row means
// [2, H, T] float32 after the dW partials.
size_t mu_bytes(const qkvp_dims* d) { return (static_cast<size_t>(2) * d->H * d->T * sizeof(float) + 15) / 16 * 16; }
size_t ws_bytes_for(const qkvp_dims* d) { return ws_bytes_for_shape(dw_shape(d)) + mu_bytes(d); }

// Split count for the dW GEMM: the fewest splits whose units fill the
// workers (SMs, or SM pairs) in whole waves to >= 90%, with at least 4
// k-blocks per split.
int choose_splits(int tiles, int kblocks, int sms) {
  int best = 1;
  double best_eff = 0.0;
  const int smax = std::max(1, std::min(kMaxSplits, kblocks / 4));
  for (int s = 1; s <= smax; ++s) {
    const int units = tiles * s;
    const int waves = (units + sms - 1) / sms;
    const double eff = static_cast<double>(units) / (static_cast<double>(waves) * sms);
    if (eff >= 0.9) return s;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

DevStatus dev_status(void* ws) { return DevStatus{static_cast<int*>(ws), g_timeout_ns}; }

// Optional kernel-boundary events (qkvp_set_timing_events).
struct TimingHook {
  cudaEvent_t ev[256];
  int n = 0, next = 0;
} g_timing;

}  // namespace

// Recorded as an external event node when the stream is being captured into
// a CUDA graph (so the graph's launches record it too), plainly otherwise.
void qkvp::mark(cudaStream_t s) {
  if (g_timing.next >= g_timing.n) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  cudaEvent_t ev = g_timing.ev[g_timing.next++];
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

namespace {

#define QKVP_TRY_CUDA(expr)                          \
  do {                                               \
    if ((expr) != cudaSuccess) return QKVP_ERR_CUDA; \
  } while (0)

// The grid barrier of the fused activation quantiser, inside the status area
// at the start of a workspace (zeroed by qkvp_workspace_init).
GridBar* grid_bar(void* ws) { return reinterpret_cast<GridBar*>(static_cast<uint8_t*>(ws) + 128); }

// Per-tensor quantisation of a bf16 activation of n elements (n % 16 == 0):
// amax, then codes and the scale, in one launch (`parts` holds one partial per
// block, up to kMaxFusedBlocks <= kMaxParts).
int quantize_activation(const uint16_t* x, int64_t n, uint8_t* x8, float* parts, float* scale, void* ws,
                        cudaStream_t s) {
  static_assert(kMaxFusedBlocks <= kMaxParts, "partials buffer too small");
  mark(s);
  QKVP_TRY_CUDA(launch_x_amax_quant(x, n, x8, parts, scale, grid_bar(ws), dev_status(ws), s));
  mark(s);
  return QKVP_OK;
}

// out [T, Nout] bf16 = epilogue((A8 [T, K] . B8 [Nout, K]^T) * sa * sb), both
// operands K-major codes (the dX GEMM body).  K and Nout multiples of 128.
// With EPI_RELU2 / EPI_DRELU2 the GEMM also writes amax partials, whose count
// lands in *nparts.
int gemm_nt(int T, int Nout, int K, const uint8_t* A8, const uint8_t* B8, const float* sa, const float* sb,
            uint16_t* out, DevStatus st, int sms, cudaStream_t s, int mode = EPI_PLAIN, float* amax_parts = nullptr,
            const uint8_t* aux8 = nullptr, const float* aux_scale = nullptr, int* nparts = nullptr) {
  const int bn = Nout % 256 == 0 ? 256 : 128;   // one box per stage: the whole B tile (this CTA's half on pairs)
  const int pair = (g_pair_mask & 2) ? 2 : 1;
  CUtensorMap tm_a, tm_b, tm_out;
  bool ok = map2d(&tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A8, K, T, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map2d(&tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B8, K, Nout, K, 128, bn / pair, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map2d(&tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, Nout, T, Nout * 2ull, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return QKVP_ERR_CUDA;
  DxParams gp;
  gp.T = T;
  gp.D = Nout;
  gp.bn = bn;
  gp.n_tiles = Nout / bn;
  gp.pair = pair;
  gp.num_units = ((T + 127) / 128 + pair - 1) / pair * gp.n_tiles;
  gp.kblocks = (K + 127) / 128;
  gp.dy_scale = sa;
  gp.w_scale = sb;
  gp.mode = mode;
  gp.amax_parts = amax_parts;
  gp.aux8 = aux8;
  gp.aux_scale = aux_scale;
  int grid = 0;
  QKVP_TRY_CUDA(launch_dx_gemm(tm_a, tm_b, tm_out, gp, sms, st, s, &grid));
  if (nparts) *nparts = grid * dx_epi_warps(mode);
  mark(s);
  return QKVP_OK;
}

// dW [R, C] bf16 = (G8 [T, R]^T . X8 [T, C]) * sg * sx, both operands read
// MN-major (token-major codes as stored), split over the tokens; partials and
// in the workspace (`ds` describes their layout), summed by a second kernel.
int gemm_tn_split(int T, int R, int C, const DwShape& ds, const uint8_t* G8, const uint8_t* X8, const float* sg,
                  const float* sx, uint16_t* dW, float* partials, DevStatus st, int sms,
                  cudaStream_t s) {
  CUtensorMap tm_g, tm_x;
  bool ok = map2d(&tm_g, CU_TENSOR_MAP_DATA_TYPE_UINT8, G8, R, T, R, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, X8, C, T, C, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return QKVP_ERR_CUDA;
  DwParams wp;
  wp.N = R;
  wp.D = C;
  wp.bn = ds.bn;
  wp.m_tiles = ds.m_tiles;
  wp.n_tiles = ds.n_tiles;
  wp.kblocks_total = ds.kblocks_total;
  // pairs split the 256 columns of a tile: one 128-column box of X8 each
  wp.pair = ((g_pair_mask & 4) && ds.bn == 256) ? 2 : 1;
  const int pair_tiles = (ds.m_tiles + wp.pair - 1) / wp.pair * ds.n_tiles;
  wp.splits = choose_splits(pair_tiles, ds.kblocks_total, sms / wp.pair);
  wp.num_units = wp.splits * pair_tiles;
  wp.partials = partials;
  wp.dy_scale = sg;
  wp.x_scale = sx;
  wp.dW = dW;
  QKVP_TRY_CUDA(launch_dw_gemm(tm_g, tm_x, wp, sms, st, s));
  mark(s);
  return QKVP_OK;
}

}  // namespace

extern "C" {

const char* qkvp_status_string(int status) {
  switch (status) {
    case QKVP_OK: return "QKVP_OK";
    case QKVP_ERR_INVALID_ARGUMENT: return "QKVP_ERR_INVALID_ARGUMENT";
    case QKVP_ERR_UNSUPPORTED: return "QKVP_ERR_UNSUPPORTED";
    case QKVP_ERR_MISALIGNED: return "QKVP_ERR_MISALIGNED";
    case QKVP_ERR_WORKSPACE_TOO_SMALL: return "QKVP_ERR_WORKSPACE_TOO_SMALL";
    case QKVP_ERR_CUDA: return "QKVP_ERR_CUDA";
    case QKVP_ERR_TIMEOUT: return "QKVP_ERR_TIMEOUT";
    case QKVP_ERR_DEVICE_INPUT: return "QKVP_ERR_DEVICE_INPUT";
    default: return "QKVP_ERR_UNKNOWN";
  }
}

size_t qkvp_workspace_bytes(const qkvp_dims* dims) {
  if (check_dims(dims) != QKVP_OK) return 0;
  return ws_bytes_for(dims);
}

size_t qkvp_bank_workspace_bytes(int L, int D, int H, int d_qk, int d_v) {
  const qkvp_dims d{1, D, H, d_qk, d_v};
  if (L < 1 || L > kMaxLayers || check_dims(&d) != QKVP_OK) return 0;
  return kStatusBytes + sizeof(BankSync);
}

int qkvp_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kStatusBytes) return QKVP_ERR_INVALID_ARGUMENT;
  QKVP_TRY_CUDA(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
  return QKVP_OK;
}

int qkvp_poll_device_status(void* ws, int* where, void* stream) {
  if (!ws) return QKVP_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host[2] = {0, 0};
  QKVP_TRY_CUDA(cudaMemcpyAsync(host, ws, sizeof(host), cudaMemcpyDeviceToHost, s));
  QKVP_TRY_CUDA(cudaMemsetAsync(ws, 0, sizeof(host), s));
  QKVP_TRY_CUDA(cudaStreamSynchronize(s));
  if (where) *where = host[1];
  return host[0];
}

int qkvp_set_timing_events(void* const* events, int n) {
  if (n < 0 || n > 256 || (n > 0 && !events)) return QKVP_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n; ++i) g_timing.ev[i] = static_cast<cudaEvent_t>(events[i]);
  g_timing.n = n;
  g_timing.next = 0;
  return QKVP_OK;
}

int qkvp_timing_events_recorded(void) { return g_timing.next; }

int qkvp_set_cta_pairs(int mask) {
  if (mask < 0 || mask > 7) return -1;
  const int prev = g_pair_mask;
  g_pair_mask = mask;
  return prev;
}

int qkvp_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000000ull || ns > 60000000000ull) return QKVP_ERR_INVALID_ARGUMENT;
  g_timeout_ns = ns;
  return QKVP_OK;
}

int qkvp_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned timeout_us, void* stream) {
  if (!ws || ws_bytes < kStatusBytes || timeout_us < 1 || timeout_us > 1000000) return QKVP_ERR_INVALID_ARGUMENT;
  if (!aligned16(ws)) return QKVP_ERR_MISALIGNED;
  DevStatus st{static_cast<int*>(ws), static_cast<uint64_t>(timeout_us) * 1000ull};
  QKVP_TRY_CUDA(launch_selftest_wait(st, static_cast<cudaStream_t>(stream)));
  return QKVP_OK;
}

int qkvp_build_rope_table(float* table, int max_pos, int d_qk, double base, void* stream) {
  if (!table || max_pos < 1 || !(base > 1.0)) return QKVP_ERR_INVALID_ARGUMENT;
  if (d_qk != 64 && d_qk != 96 && d_qk != 128) return QKVP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_pos) * d_qk > (int64_t(1) << 31)) return QKVP_ERR_UNSUPPORTED;
  if (!aligned16(table)) return QKVP_ERR_MISALIGNED;
  QKVP_TRY_CUDA(launch_rope_table(table, max_pos, d_qk, base, static_cast<cudaStream_t>(stream)));
  return QKVP_OK;
}

int qkvp_quantize_bank(int L, int D, int H, int d_qk, int d_v, const uint16_t* const* Wq,
                       const uint16_t* const* Wk, const uint16_t* const* Wv, uint8_t* W8, uint8_t* W8T,
                       float* w_scale, void* ws, size_t ws_bytes, void* stream) {
  const qkvp_dims d{1, D, H, d_qk, d_v};
  if (L < 1 || !Wq || !Wk || !Wv || !W8 || !W8T || !w_scale || !ws) return QKVP_ERR_INVALID_ARGUMENT;
  const int rc = check_dims(&d);
  if (rc != QKVP_OK) return rc;
  if (L > kMaxLayers) return QKVP_ERR_UNSUPPORTED;
  BankArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int l = 0; l < L; ++l) {
    if (!Wq[l] || !Wk[l] || !Wv[l]) return QKVP_ERR_INVALID_ARGUMENT;
    if (!aligned16(Wq[l]) || !aligned16(Wk[l]) || !aligned16(Wv[l])) return QKVP_ERR_MISALIGNED;
    a.Wq[l] = Wq[l];
    a.Wk[l] = Wk[l];
    a.Wv[l] = Wv[l];
  }
  if (!aligned16(W8) || !aligned16(W8T) || !aligned16(w_scale) || !aligned16(ws)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < qkvp_bank_workspace_bytes(L, D, H, d_qk, d_v)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  a.W8 = W8;
  a.W8T = W8T;
  a.w_scale = w_scale;
  a.L = L;
  a.D = D;
  a.Nq = H * d_qk;
  a.N = H * (2 * d_qk + d_v);
  BankSync* sy = reinterpret_cast<BankSync*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mark(s);
  QKVP_TRY_CUDA(launch_bank_refresh(a, sy, dev_status(ws), s));
  mark(s);
  return QKVP_OK;
}

namespace {
// The packed GEMM with its fused epilogue, from x8 and its scale (arguments
// already validated).
// Slots of a token block in the order q, v, k tiles are interleaved in
// proportion to their counts: tile i of a list of n sits at (2i + 1) / 2n,
// ties in the order q, v, k (nq = nv = 3 gives q0 v0 k0 q1 v1 k1 q2 v2 k2).
static void fwd_tile_order(FwdParams& p) {
  const int first[3] = {0, 2 * p.nq, p.nq};   // q, v, k tiles
  const int count[3] = {p.nq, p.nv, p.nq};
  int next[3] = {0, 0, 0};
  for (int slot = 0; slot < p.n_tiles; ++slot) {
    int best = -1;
    for (int l = 0; l < 3; ++l) {
      if (next[l] >= count[l]) continue;
      // compare (2 next[l] + 1) / count[l] across lists without division
      if (best < 0 || static_cast<int64_t>(2 * next[l] + 1) * count[best] <
                          static_cast<int64_t>(2 * next[best] + 1) * count[l])
        best = l;
    }
    p.tile_order[slot] = static_cast<uint8_t>(first[best] + next[best]++);
  }
}

int forward_gemm(const qkvp_dims* dims, float eps, const float* rope_table, int max_pos, const uint8_t* x8,
                 const float* x_scale, const int32_t* pos, const uint8_t* W8, const float* w_scale, uint16_t* q,
                 uint16_t* k, uint16_t* v, float* rstd, void* ws, int sms, cudaStream_t s) {
  const int T = dims->T, D = dims->D, H = dims->H, dqk = dims->d_qk, dv = dims->d_v;
  const int N = H * (2 * dqk + dv);
  const int tiles = (T + 127) / 128;
  // Tiles of the packed GEMM cover whole heads: q/k tiles of hq heads (the
  // last one may hold fewer), v tiles of 2 heads.  Each stage loads B as one
  // box of the full tile height, hq*d_qk rows (q/k) or 2*d_v rows (v), or
  // on CTA pairs each CTA half of it.
  const int hq = dqk == 64 ? 4 : 2;
  const int pair = (g_pair_mask & 1) ? 2 : 1;
  CUtensorMap tm_x8, tm_w, tm_wv, tm_q, tm_k, tm_v;
  bool ok = map2d(&tm_x8, CU_TENSOR_MAP_DATA_TYPE_UINT8, x8, D, T, D, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, W8, D, N, D, 128, hq * dqk / pair,
                   CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map2d(&tm_wv, CU_TENSOR_MAP_DATA_TYPE_UINT8, W8, D, N, D, 128, 2 * dv / pair, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map3d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, dqk, T, H, 64, 32, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map3d(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, dqk, T, H, 64, 32, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && map3d(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v, dv, T, H, 64, 32, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return QKVP_ERR_CUDA;
  FwdParams p;
  p.T = T;
  p.H = H;
  p.d_qk = dqk;
  p.d_v = dv;
  p.hq = hq;
  p.nq = (H + p.hq - 1) / p.hq;
  p.nv = (H + 1) / 2;
  p.n_tiles = 2 * p.nq + p.nv;
  fwd_tile_order(p);
  p.pair = pair;
  p.num_units = (tiles + pair - 1) / pair * p.n_tiles;
  p.kblocks = D / 128;
  p.eps = eps;
  p.x_scale = x_scale;
  p.w_scale = w_scale;
  p.rope = rope_table;
  p.max_pos = max_pos;
  p.pos = pos;
  p.rstd = rstd;
  QKVP_TRY_CUDA(launch_fwd_gemm(tm_x8, tm_w, tm_wv, tm_q, tm_k, tm_v, p, sms, dev_status(ws), s));
  mark(s);
  return QKVP_OK;
}
}  // namespace

int qkvp_forward(const qkvp_dims* dims, float eps, const float* rope_table, int max_pos, const uint16_t* x,
                 const int32_t* pos, const uint8_t* W8, const float* w_scale, uint16_t* q, uint16_t* k,
                 uint16_t* v, float* rstd, uint8_t* x8, float* x_scale, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_dims(dims);
  if (rc != QKVP_OK) return rc;
  if (!rope_table || !x || !pos || !W8 || !w_scale || !q || !k || !v || !rstd || !x8 || !x_scale || !ws)
    return QKVP_ERR_INVALID_ARGUMENT;
  if (max_pos < 1 || !(eps >= 0.f) || !(eps < 1.f)) return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {rope_table, x, pos, W8, w_scale, q, k, v, rstd, x8, x_scale, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < ws_bytes_for(dims)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* xparts = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  rc = quantize_activation(x, static_cast<int64_t>(dims->T) * dims->D, x8, xparts, x_scale, ws, s);
  if (rc != QKVP_OK) return rc;
  return forward_gemm(dims, eps, rope_table, max_pos, x8, x_scale, pos, W8, w_scale, q, k, v, rstd, ws, sms, s);
}

size_t qkvp_activation_workspace_bytes(void) { return kStatusBytes + kPartsBytes; }

int qkvp_quantize_activation(const uint16_t* x, int64_t n, uint8_t* x8, float* x_scale, void* ws, size_t ws_bytes,
                             void* stream) {
  if (!x || !x8 || !x_scale || !ws || n < 1) return QKVP_ERR_INVALID_ARGUMENT;
  if (n % 16 != 0 || n > (int64_t(1) << 40)) return QKVP_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(x8) || !aligned16(x_scale) || !aligned16(ws)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < qkvp_activation_workspace_bytes()) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  float* parts = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  return quantize_activation(x, n, x8, parts, x_scale, ws, static_cast<cudaStream_t>(stream));
}

int qkvp_forward_quantized(const qkvp_dims* dims, float eps, const float* rope_table, int max_pos, const uint8_t* x8,
                           const float* x_scale, const int32_t* pos, const uint8_t* W8, const float* w_scale,
                           uint16_t* q, uint16_t* k, uint16_t* v, float* rstd, void* ws, size_t ws_bytes,
                           void* stream) {
  int rc = check_dims(dims);
  if (rc != QKVP_OK) return rc;
  if (!rope_table || !x8 || !x_scale || !pos || !W8 || !w_scale || !q || !k || !v || !rstd || !ws)
    return QKVP_ERR_INVALID_ARGUMENT;
  if (max_pos < 1 || !(eps >= 0.f) || !(eps < 1.f)) return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {rope_table, x8, x_scale, pos, W8, w_scale, q, k, v, rstd, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < ws_bytes_for(dims)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mark(s);
  return forward_gemm(dims, eps, rope_table, max_pos, x8, x_scale, pos, W8, w_scale, q, k, v, rstd, ws, sms, s);
}

int qkvp_backward(const qkvp_dims* dims, const float* rope_table, int max_pos, const uint16_t* dq,
                  const uint16_t* dk, const uint16_t* dv, const uint16_t* q, const uint16_t* k, const float* rstd,
                  const int32_t* pos, const uint8_t* W8T, const float* w_scale, const uint8_t* x8,
                  const float* x_scale, uint16_t* dx, uint16_t* dW, uint8_t* dY8, float* dy_scale, void* ws,
                  size_t ws_bytes, void* stream) {
  int rc = check_dims(dims);
  if (rc != QKVP_OK) return rc;
  if (!rope_table || !dq || !dk || !dv || !q || !k || !rstd || !pos || !W8T || !w_scale || !x8 || !x_scale || !dx ||
      !dW || !dY8 || !dy_scale || !ws)
    return QKVP_ERR_INVALID_ARGUMENT;
  if (max_pos < 1) return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {rope_table, dq, dk, dv, q, k, rstd, pos, W8T, w_scale, x8, x_scale, dx, dW, dY8,
                        dy_scale, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < ws_bytes_for(dims)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;

  const int T = dims->T, D = dims->D, H = dims->H, dqk = dims->d_qk, dvw = dims->d_v;
  const int N = H * (2 * dqk + dvw);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* dyparts = reinterpret_cast<float*>(wsb + kStatusBytes + kPartsBytes);
  float* dwparts = reinterpret_cast<float*>(wsb + kStatusBytes + 2 * kPartsBytes);
  float* mu = reinterpret_cast<float*>(wsb + ws_bytes_for_shape(dw_shape(dims)));
  const DevStatus st = dev_status(ws);

  BwdMaps m;
  constexpr uint32_t R = kBwdUnitRows;
  bool ok = map3d(&m.dq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dq, dqk, T, H, 32, R, 1, CU_TENSOR_MAP_SWIZZLE_64B);
  ok = ok && map3d(&m.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, dqk, T, H, 32, R, 1, CU_TENSOR_MAP_SWIZZLE_64B);
  ok = ok && map3d(&m.dk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dk, dqk, T, H, 32, R, 1, CU_TENSOR_MAP_SWIZZLE_64B);
  ok = ok && map3d(&m.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, dqk, T, H, 32, R, 1, CU_TENSOR_MAP_SWIZZLE_64B);
  ok = ok && map3d(&m.dv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dv, dvw, T, H, 32, R, 1, CU_TENSOR_MAP_SWIZZLE_64B);
  ok = ok && map2d(&m.dy8, CU_TENSOR_MAP_DATA_TYPE_UINT8, dY8, N, T, N, 32, R, CU_TENSOR_MAP_SWIZZLE_32B);
  if (!ok) return QKVP_ERR_CUDA;

  BwdParams bp;
  bp.T = T;
  bp.H = H;
  bp.d_qk = dqk;
  bp.d_v = dvw;
  bp.N = N;
  bp.tiles = (T + kBwdUnitRows - 1) / kBwdUnitRows;
  bp.num_units = bp.tiles * H * 3;
  bp.rstd = rstd;
  bp.pos = pos;
  bp.rope = rope_table;
  bp.max_pos = max_pos;
  bp.partials = dyparts;
  bp.nparts = std::min({bp.num_units, sms, kMaxParts});
  bp.dy_scale = dy_scale;
  bp.mu = mu;
  mark(s);
  QKVP_TRY_CUDA(launch_bwd_amax(m, bp, bp.nparts, st, s));
  mark(s);
  QKVP_TRY_CUDA(launch_bwd_quant(m, bp, std::min(bp.num_units, sms), st, s));
  mark(s);

  // dX [T, D] = dY8 [T, N] . W8 with the cached W8T [D, N] as the K-major operand
  rc = gemm_nt(T, D, N, dY8, W8T, dy_scale, w_scale, dx, st, sms, s);
  if (rc != QKVP_OK) return rc;
  // dW [N, D] = dY8^T . x8, both read MN-major
  rc = gemm_tn_split(T, N, D, dw_shape(dims), dY8, x8, dy_scale, x_scale, dW, dwparts, st, sms, s);
  if (rc != QKVP_OK) return rc;
  return QKVP_OK;
}

// ---------------------------------------------------------------------------
// Weight refresh for single matrices and the O projection over the V/O bank
// ---------------------------------------------------------------------------
size_t qkvp_weight_workspace_bytes(int L, int R, int C) {
  if (L < 1 || L > kMaxLayers || R < 128 || C < 128 || R % 128 || C % 128 || R > 65536 || C > 16384) return 0;
  return kStatusBytes + sizeof(BankSync);
}

int qkvp_quantize_weight(int L, int R, int C, const uint16_t* const* W, uint8_t* W8, uint8_t* W8T, float* w_scale,
                         void* ws, size_t ws_bytes, void* stream) {
  if (L < 1 || !W || !W8 || !W8T || !w_scale || !ws || R < 1 || C < 1) return QKVP_ERR_INVALID_ARGUMENT;
  const size_t need = qkvp_weight_workspace_bytes(L, R, C);
  if (need == 0) return QKVP_ERR_UNSUPPORTED;
  // the bank kernels with empty Q and K packs: every row comes from W[l]
  BankArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int l = 0; l < L; ++l) {
    if (!W[l]) return QKVP_ERR_INVALID_ARGUMENT;
    if (!aligned16(W[l])) return QKVP_ERR_MISALIGNED;
    a.Wq[l] = a.Wk[l] = a.Wv[l] = W[l];
  }
  if (!aligned16(W8) || !aligned16(W8T) || !aligned16(w_scale) || !aligned16(ws)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < need) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  a.W8 = W8;
  a.W8T = W8T;
  a.w_scale = w_scale;
  a.L = L;
  a.D = C;
  a.Nq = 0;
  a.N = R;
  BankSync* sy = reinterpret_cast<BankSync*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mark(s);
  QKVP_TRY_CUDA(launch_bank_refresh(a, sy, dev_status(ws), s));
  mark(s);
  return QKVP_OK;
}

namespace {
int check_oproj(int T, int D, int K) {
  if (T < 1 || D < 1 || K < 1) return QKVP_ERR_INVALID_ARGUMENT;
  if (T > (1 << 24) || D % 128 || K % 128 || D > 16384 || K > 16384) return QKVP_ERR_UNSUPPORTED;
  return QKVP_OK;
}
}  // namespace

size_t qkvp_oproj_workspace_bytes(int T, int D, int K) {
  if (check_oproj(T, D, K) != QKVP_OK) return 0;
  return ws_bytes_for_shape(dw_shape_rc(D, K, T));
}

int qkvp_oproj_forward(int T, int D, int K, const uint16_t* a, const uint8_t* Wo8, const float* wo_scale,
                       uint16_t* out, uint8_t* a8, float* a_scale, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_oproj(T, D, K);
  if (rc != QKVP_OK) return rc;
  if (!a || !Wo8 || !wo_scale || !out || !a8 || !a_scale || !ws) return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {a, Wo8, wo_scale, out, a8, a_scale, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < qkvp_oproj_workspace_bytes(T, D, K)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* aparts = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kStatusBytes);
  rc = quantize_activation(a, static_cast<int64_t>(T) * K, a8, aparts, a_scale, ws, s);
  if (rc != QKVP_OK) return rc;
  // out [T, D] = a8 [T, K] . Wo8 [D, K]^T
  return gemm_nt(T, D, K, a8, Wo8, a_scale, wo_scale, out, dev_status(ws), sms, s);
}

int qkvp_oproj_backward(int T, int D, int K, const uint16_t* dout, const uint8_t* Wo8T, const float* wo_scale,
                        const uint8_t* a8, const float* a_scale, uint16_t* da, uint16_t* dWo, uint8_t* dout8,
                        float* dout_scale, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_oproj(T, D, K);
  if (rc != QKVP_OK) return rc;
  if (!dout || !Wo8T || !wo_scale || !a8 || !a_scale || !da || !dWo || !dout8 || !dout_scale || !ws)
    return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {dout, Wo8T, wo_scale, a8, a_scale, da, dWo, dout8, dout_scale, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < qkvp_oproj_workspace_bytes(T, D, K)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* gparts = reinterpret_cast<float*>(wsb + kStatusBytes + kPartsBytes);
  const DwShape ds = dw_shape_rc(D, K, T);
  float* dwparts = reinterpret_cast<float*>(wsb + kStatusBytes + 2 * kPartsBytes);
  const DevStatus st = dev_status(ws);
  rc = quantize_activation(dout, static_cast<int64_t>(T) * D, dout8, gparts, dout_scale, ws, s);
  if (rc != QKVP_OK) return rc;
  // da [T, K] = dout8 [T, D] . Wo8 with the cached Wo8T [K, D] as the K-major operand
  rc = gemm_nt(T, K, D, dout8, Wo8T, dout_scale, wo_scale, da, st, sms, s);
  if (rc != QKVP_OK) return rc;
  // dWo [D, K] = dout8^T . a8, both read MN-major
  return gemm_tn_split(T, D, K, ds, dout8, a8, dout_scale, a_scale, dWo, dwparts, st, sms, s);
}

// ---------------------------------------------------------------------------
// FP8 ReLU-squared MLP
// ---------------------------------------------------------------------------
namespace {
int check_mlp(int T, int D, int F) {
  if (T < 1 || D < 1 || F < 1) return QKVP_ERR_INVALID_ARGUMENT;
  if (T > (1 << 24) || D % 128 || F % 128 || D > 16384 || F > 65536) return QKVP_ERR_UNSUPPORTED;
  return QKVP_OK;
}
// both weight gradients share the partials (they run one after the other)
size_t mlp_ws_bytes(int T, int D, int F) {
  return kStatusBytes + 2 * kPartsBytes +
         std::max(dw_partial_bytes(dw_shape_rc(F, D, T), kMaxSplits), dw_partial_bytes(dw_shape_rc(D, F, T), kMaxSplits));
}
// h, dpre: bf16 intermediates quantised from the GEMM's own amax partials
int quantize_from_parts(const uint16_t* v, int64_t n, uint8_t* v8, const float* parts, int nparts, float* scale,
                        int sms, cudaStream_t s) {
  if (nparts < 1 || nparts > kMaxParts) return QKVP_ERR_CUDA;
  QKVP_TRY_CUDA(launch_x_quant(v, n, v8, parts, nparts, scale, 4 * sms, s));
  mark(s);
  return QKVP_OK;
}
}  // namespace

size_t qkvp_mlp_workspace_bytes(int T, int D, int F) {
  if (check_mlp(T, D, F) != QKVP_OK) return 0;
  return mlp_ws_bytes(T, D, F);
}

int qkvp_mlp_forward(int T, int D, int F, const uint16_t* x, const uint8_t* W1_8, const float* w1_scale,
                     const uint8_t* W2_8, const float* w2_scale, uint16_t* out, uint8_t* x8, float* x_scale,
                     uint16_t* h, uint8_t* h8, float* h_scale, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_mlp(T, D, F);
  if (rc != QKVP_OK) return rc;
  if (!x || !W1_8 || !w1_scale || !W2_8 || !w2_scale || !out || !x8 || !x_scale || !h || !h8 || !h_scale || !ws)
    return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {x, W1_8, w1_scale, W2_8, w2_scale, out, x8, x_scale, h, h8, h_scale, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < mlp_ws_bytes(T, D, F)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* parts_a = reinterpret_cast<float*>(wsb + kStatusBytes);
  float* parts_b = reinterpret_cast<float*>(wsb + kStatusBytes + kPartsBytes);
  const DevStatus st = dev_status(ws);
  rc = quantize_activation(x, static_cast<int64_t>(T) * D, x8, parts_a, x_scale, ws, s);
  if (rc != QKVP_OK) return rc;
  // h [T, F] = relu(x8 . W1_8^T * s_x * s_1)^2 in bf16, with its amax partials
  int nparts = 0;
  rc = gemm_nt(T, F, D, x8, W1_8, x_scale, w1_scale, h, st, sms, s, EPI_RELU2, parts_b, nullptr, nullptr, &nparts);
  if (rc != QKVP_OK) return rc;
  rc = quantize_from_parts(h, static_cast<int64_t>(T) * F, h8, parts_b, nparts, h_scale, sms, s);
  if (rc != QKVP_OK) return rc;
  // out [T, D] = h8 . W2_8^T * s_h * s_2
  return gemm_nt(T, D, F, h8, W2_8, h_scale, w2_scale, out, st, sms, s);
}

int qkvp_mlp_backward(int T, int D, int F, const uint16_t* dout, const uint8_t* W1_8T, const float* w1_scale,
                      const uint8_t* W2_8T, const float* w2_scale, const uint8_t* x8, const float* x_scale,
                      const uint8_t* h8, const float* h_scale, uint16_t* dx, uint16_t* dW1, uint16_t* dW2,
                      uint8_t* dout8, float* dout_scale, uint16_t* dpre, uint8_t* dpre8, float* dpre_scale, void* ws,
                      size_t ws_bytes, void* stream) {
  int rc = check_mlp(T, D, F);
  if (rc != QKVP_OK) return rc;
  if (!dout || !W1_8T || !w1_scale || !W2_8T || !w2_scale || !x8 || !x_scale || !h8 || !h_scale || !dx || !dW1 ||
      !dW2 || !dout8 || !dout_scale || !dpre || !dpre8 || !dpre_scale || !ws)
    return QKVP_ERR_INVALID_ARGUMENT;
  const void* ptrs[] = {dout, W1_8T, w1_scale, W2_8T, w2_scale, x8, x_scale, h8, h_scale, dx, dW1, dW2, dout8,
                        dout_scale, dpre, dpre8, dpre_scale, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return QKVP_ERR_MISALIGNED;
  if (ws_bytes < mlp_ws_bytes(T, D, F)) return QKVP_ERR_WORKSPACE_TOO_SMALL;
  const int sms = sm_count();
  if (sms <= 0) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* parts_a = reinterpret_cast<float*>(wsb + kStatusBytes);
  float* parts_b = reinterpret_cast<float*>(wsb + kStatusBytes + kPartsBytes);
  float* dwparts = reinterpret_cast<float*>(wsb + kStatusBytes + 2 * kPartsBytes);
  const DevStatus st = dev_status(ws);
  rc = quantize_activation(dout, static_cast<int64_t>(T) * D, dout8, parts_a, dout_scale, ws, s);
  if (rc != QKVP_OK) return rc;
  // dpre [T, F] = (dout8 . W2_8 * s_g * s_2) * 2 sqrt(h8 * s_h), via the cached W2_8T [F, D]
  int nparts = 0;
  rc = gemm_nt(T, F, D, dout8, W2_8T, dout_scale, w2_scale, dpre, st, sms, s, EPI_DRELU2, parts_b, h8, h_scale,
               &nparts);
  if (rc != QKVP_OK) return rc;
  rc = quantize_from_parts(dpre, static_cast<int64_t>(T) * F, dpre8, parts_b, nparts, dpre_scale, sms, s);
  if (rc != QKVP_OK) return rc;
  // dx [T, D] = dpre8 . W1_8 * s_p * s_1, via the cached W1_8T [D, F]
  rc = gemm_nt(T, D, F, dpre8, W1_8T, dpre_scale, w1_scale, dx, st, sms, s);
  if (rc != QKVP_OK) return rc;
  // dW1 [F, D] = dpre8^T . x8;  dW2 [D, F] = dout8^T . h8  (both operands MN-major)
  rc = gemm_tn_split(T, F, D, dw_shape_rc(F, D, T), dpre8, x8, dpre_scale, x_scale, dW1, dwparts, st, sms, s);
  if (rc != QKVP_OK) return rc;
  return gemm_tn_split(T, D, F, dw_shape_rc(D, F, T), dout8, h8, dout_scale, h_scale, dW2, dwparts, st, sms, s);
}

}  // extern "C"

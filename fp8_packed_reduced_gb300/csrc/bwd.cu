// Backward of the fused epilogue (RoPE, per-head RMSNorm, split) and the FP8
// quantisation of its result dY, in two bandwidth-bound passes:
//   pass 1 (amax)   recompute dY, keep only its per-tensor amax
//   pass 2 (quant)  recompute dY, quantise with s_dy = amax/448 and write
//                   dY8 [T, N] and dY8T [N, Tp] from the one read
// Recomputing in pass 2 moves fewer bytes than storing a bf16 dY in pass 1
// and reading it back.
//
// For one (token, head) of q (likewise k), with the saved output o = q_out,
// the upstream gradient g_out = dq and the saved r = rstd:
//   y  = RoPE^T(o),  g = RoPE^T(g_out),  mu = mean(g * y) = mean(g_out * o)
//   dY = r * (g - y * mu) = r * RoPE^T(g_out - mu * o)
// (RoPE is a rotation, so the inner product needs no rotation and one
// inverse rotation of (g_out - mu * o) suffices).  dY_v = dv.
//
// Work unit: 128 tokens x one head x one part (q, k or v).  One thread per
// token row; the inputs arrive by TMA as 32-column boxes with 64-byte
// swizzling, which the row-per-thread reads access without bank conflicts.
#include "kernels.cuh"

namespace qkvp {

constexpr int kInBox = 8192;     // 128 rows x 32 bf16
constexpr int kOutBox = 4096;    // 128 x 32 codes
constexpr int kBwdAmaxSmem = 1024 + 8 * kInBox;
constexpr int kBwdQuantSmem = 1024 + 8 * kInBox + 8 * kOutBox;

struct BwdUnit {
  int part, h, t0, col0;
};

__device__ __forceinline__ BwdUnit bwd_decode(const BwdParams& p, int u) {
  BwdUnit b;
  b.part = u % 3;
  b.h = (u / 3) % p.H;
  b.t0 = (u / (3 * p.H)) * 128;
  b.col0 = b.part == 0 ? b.h * p.d_qk : b.part == 1 ? (p.H + b.h) * p.d_qk : 2 * p.H * p.d_qk + b.h * p.d_v;
  return b;
}

// Thread 0: expect the bytes and issue the TMA loads of unit b.
__device__ __forceinline__ void bwd_issue_loads(const BwdMaps& m, const BwdParams& p, const BwdUnit& b,
                                                uint8_t* in0, uint8_t* in1, uint64_t* bar) {
  const int d = b.part < 2 ? p.d_qk : p.d_v;
  const int nbox = d / 32;
  mbar_arrive_expect_tx(bar, static_cast<uint32_t>((b.part < 2 ? 2 : 1) * nbox * kInBox));
  const CUtensorMap* g = b.part == 0 ? &m.dq : b.part == 1 ? &m.dk : &m.dv;
  for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + j * kInBox, g, bar, 32 * j, b.t0, b.h);
  if (b.part < 2) {
    const CUtensorMap* o = b.part == 0 ? &m.q : &m.k;
    for (int j = 0; j < nbox; ++j) tma_load_3d(in1 + j * kInBox, o, bar, 32 * j, b.t0, b.h);
  }
}

// 16 consecutive bf16 values of row r starting at column c0 (c0 % 16 == 0).
__device__ __forceinline__ void load16(const uint8_t* boxes, int r, int c0, float (&v)[16], bool valid) {
  const uint8_t* box = boxes + (c0 >> 5) * kInBox + r * 64;
  const int cc = (c0 & 31) >> 3;
  const uint4 x0 = *reinterpret_cast<const uint4*>(box + ((cc ^ ((r >> 1) & 3)) << 4));
  const uint4 x1 = *reinterpret_cast<const uint4*>(box + (((cc + 1) ^ ((r >> 1) & 3)) << 4));
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = valid ? bf16_lo(w[i]) : 0.f;
    v[2 * i + 1] = valid ? bf16_hi(w[i]) : 0.f;
  }
}

// mean(g_out * o) over row r of a q/k unit, streamed from shared memory.
template <int DQK>
__device__ __forceinline__ float row_mean_dot(const uint8_t* in0, const uint8_t* in1, int r) {
  float dot = 0.f;
#pragma unroll 2
  for (int c0 = 0; c0 < DQK; c0 += 16) {
    float g[16], o[16];
    load16(in0, r, c0, g, true);
    load16(in1, r, c0, o, true);
#pragma unroll
    for (int j = 0; j < 16; ++j) dot = fmaf(g[j], o[j], dot);
  }
  return __fdiv_rn(dot, static_cast<float>(DQK));
}

// dY of row r of a q or k unit, 16 pairs at a time: columns [16g, 16g+16)
// into a[] and [HALF+16g, HALF+16g+16) into b[].  Rows past T give 0.
template <int DQK>
__device__ __forceinline__ void dy_group(const uint8_t* in0, const uint8_t* in1, int r, float mu, float rstd,
                                         int pos, bool valid, int g, const BwdParams& p, float (&a)[16],
                                         float (&b)[16]) {
  constexpr int HALF = DQK / 2;
  float ga[16], gb[16], oa[16], ob[16];
  load16(in0, r, g * 16, ga, true);
  load16(in0, r, HALF + g * 16, gb, true);
  load16(in1, r, g * 16, oa, true);
  load16(in1, r, HALF + g * 16, ob, true);
  const float2* rope = reinterpret_cast<const float2*>(p.rope) + static_cast<int64_t>(g * 16) * p.max_pos + pos;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float ua = ga[j] - mu * oa[j];
    const float ub = gb[j] - mu * ob[j];
    const float2 cs = __ldg(rope + static_cast<int64_t>(j) * p.max_pos);
    a[j] = valid ? rstd * (ua * cs.x + ub * cs.y) : 0.f;
    b[j] = valid ? rstd * (ub * cs.x - ua * cs.y) : 0.f;
  }
}

// Per-row saved state of a q/k unit: rstd and position (checked).
__device__ __forceinline__ void row_state(const BwdParams& p, const BwdUnit& b, int t, bool valid, float& rstd,
                                          int& pos, const DevStatus& st, int kid) {
  rstd = 0.f;
  pos = 0;
  if (!valid) return;
  rstd = __ldg(p.rstd + (static_cast<int64_t>(b.part) * p.H + b.h) * p.T + t);
  pos = __ldg(p.pos + t);
  if (pos < 0 || pos >= p.max_pos) {
    record_error(st, QKVP_ERR_DEVICE_INPUT, kid);
    pos = 0;
  }
}

// ---------------------------------------------------------------------------
// Pass 1: amax of dY.  Persistent grid; one partial maximum per block.
// ---------------------------------------------------------------------------
template <int DQK>
__global__ void __launch_bounds__(128) bwd_amax_kernel(const __grid_constant__ BwdMaps m,
                                                       const __grid_constant__ BwdParams p, DevStatus st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* in0 = smem;
  uint8_t* in1 = smem + 4 * kInBox;
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red[32];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int r = threadIdx.x;
  float mx = 0.f;
  int it = 0;
  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
    const BwdUnit b = bwd_decode(p, u);
    if (threadIdx.x == 0) bwd_issue_loads(m, p, b, in0, in1, &bar);
    const int t = b.t0 + r;
    const bool valid = t < p.T;
    float rstd;
    int pos;
    if (b.part < 2) row_state(p, b, t, valid, rstd, pos, st, KID_BWD_AMAX);
    const bool ok = __syncthreads_and(mbar_wait(&bar, it & 1, &abort_flag, st, KID_BWD_AMAX));
    if (!ok) break;
    if (b.part < 2) {
      const float mu = row_mean_dot<DQK>(in0, in1, r);
#pragma unroll 1
      for (int g = 0; g < DQK / 32; ++g) {
        float a[16], c[16];
        dy_group<DQK>(in0, in1, r, mu, rstd, pos, valid, g, p, a, c);
#pragma unroll
        for (int j = 0; j < 16; ++j) mx = fmaxf(mx, fmaxf(fabsf(a[j]), fabsf(c[j])));
      }
    } else {
#pragma unroll 2
      for (int c0 = 0; c0 < 128; c0 += 16) {
        float v[16];
        load16(in0, r, c0, v, valid);
#pragma unroll
        for (int j = 0; j < 16; ++j) mx = fmaxf(mx, fabsf(v[j]));
      }
    }
    __syncthreads();  // inputs consumed before the next unit's loads
  }
  mx = block_max(mx, red);
  if (threadIdx.x == 0) p.partials[blockIdx.x] = mx;
}

// ---------------------------------------------------------------------------
// Pass 2: quantise dY and write both layouts.
// ---------------------------------------------------------------------------
// Codes of 16 consecutive columns [c0, c0+16) of row r into both staging
// layouts: token-major boxes [128 rows][32 codes] (plain) and column-major
// boxes [32 columns][128 tokens] (128-byte swizzle).
__device__ __forceinline__ void emit16(const float (&v)[16], float s, int r, int c0, uint8_t* out8, uint8_t* out8t) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = quant4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], s);
  *reinterpret_cast<uint4*>(out8 + (c0 >> 5) * kOutBox + r * 32 + (c0 & 31)) = make_uint4(w[0], w[1], w[2], w[3]);
  uint8_t* boxt = out8t + (c0 >> 5) * kOutBox;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int i = (c0 & 31) + j;
    boxt[i * 128 + (((r >> 4) ^ (i & 7)) << 4) + (r & 15)] = static_cast<uint8_t>(w[j >> 2] >> (8 * (j & 3)));
  }
}

template <int DQK>
__global__ void __launch_bounds__(128) bwd_quant_kernel(const __grid_constant__ BwdMaps m,
                                                        const __grid_constant__ BwdParams p, DevStatus st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* in0 = smem;
  uint8_t* in1 = smem + 4 * kInBox;
  uint8_t* out8 = smem + 8 * kInBox;
  uint8_t* out8t = out8 + 4 * kOutBox;
  __shared__ __align__(8) uint64_t bar;
  __shared__ float red[32];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const float amax = block_reduce_partials(p.partials, p.nparts, red);
  const float s = scale_from_amax(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *p.dy_scale = s;
  const int r = threadIdx.x;
  int it = 0;
  for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
    const BwdUnit b = bwd_decode(p, u);
    if (threadIdx.x == 0) {
      bulk_wait_read<0>();  // the previous unit's stores have read the staging tiles
      bwd_issue_loads(m, p, b, in0, in1, &bar);
    }
    const int t = b.t0 + r;
    const bool valid = t < p.T;
    float rstd;
    int pos;
    if (b.part < 2) row_state(p, b, t, valid, rstd, pos, st, KID_BWD_QUANT);
    const bool ok = __syncthreads_and(mbar_wait(&bar, it & 1, &abort_flag, st, KID_BWD_QUANT));
    if (!ok) break;
    int nbox;
    if (b.part < 2) {
      const float mu = row_mean_dot<DQK>(in0, in1, r);
#pragma unroll 1
      for (int g = 0; g < DQK / 32; ++g) {
        float a[16], c[16];
        dy_group<DQK>(in0, in1, r, mu, rstd, pos, valid, g, p, a, c);
        emit16(a, s, r, g * 16, out8, out8t);
        emit16(c, s, r, DQK / 2 + g * 16, out8, out8t);
      }
      nbox = DQK / 32;
    } else {
#pragma unroll 2
      for (int c0 = 0; c0 < 128; c0 += 16) {
        float v[16];
        load16(in0, r, c0, v, valid);
        emit16(v, s, r, c0, out8, out8t);
      }
      nbox = 4;
    }
    fence_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int j = 0; j < nbox; ++j) {
        tma_store_2d(&m.dy8, out8 + j * kOutBox, b.col0 + 32 * j, b.t0);
        tma_store_2d(&m.dy8t, out8t + j * kOutBox, b.t0, b.col0 + 32 * j);
      }
      bulk_commit();
    }
  }
  if (threadIdx.x == 0) bulk_wait_all<0>();
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <class K>
static cudaError_t set_smem_attr(K kernel, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done[dev] = true;
  return e;
}

template <int DQK>
static cudaError_t launch_amax_t(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  static bool done[64] = {};
  cudaError_t e = set_smem_attr(bwd_amax_kernel<DQK>, kBwdAmaxSmem, done);
  if (e != cudaSuccess) return e;
  bwd_amax_kernel<DQK><<<grid, 128, kBwdAmaxSmem, s>>>(m, p, st);
  return cudaGetLastError();
}

template <int DQK>
static cudaError_t launch_quant_t(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  static bool done[64] = {};
  cudaError_t e = set_smem_attr(bwd_quant_kernel<DQK>, kBwdQuantSmem, done);
  if (e != cudaSuccess) return e;
  bwd_quant_kernel<DQK><<<grid, 128, kBwdQuantSmem, s>>>(m, p, st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_amax(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  switch (p.d_qk) {
    case 64: return launch_amax_t<64>(m, p, grid, st, s);
    case 96: return launch_amax_t<96>(m, p, grid, st, s);
    case 128: return launch_amax_t<128>(m, p, grid, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_quant(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  switch (p.d_qk) {
    case 64: return launch_quant_t<64>(m, p, grid, st, s);
    case 96: return launch_quant_t<96>(m, p, grid, st, s);
    case 128: return launch_quant_t<128>(m, p, grid, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvp

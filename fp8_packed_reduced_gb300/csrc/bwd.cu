// Backward of the fused epilogue (RoPE, per-head RMSNorm, split) and the FP8
// quantisation of its result dY, in two bandwidth-bound passes:
//   pass 1 (amax)   recompute dY, keep only its per-tensor amax
//   pass 2 (quant)  recompute dY, quantise with s_dy = amax/448, write dY8 [T, N]
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
// Work unit: 128 tokens x one head x one part (q, k or v).  Persistent CTA
// per SM, warp-specialised:
//   warp 0      TMA producer: the unit's input boxes ([128 tokens x 32 cols],
//               64-byte swizzle) into a ring of kBwdStages stages
//   warps 1-8   two consumer groups of four warps; group g takes every other
//               unit of the CTA; one token row per thread (conflict-free reads
//               of the swizzled boxes); pass 2 stages the codes of its unit and
//               stores them by TMA while the other group computes
#include "kernels.cuh"

namespace qkvp {

constexpr int kInBox = 8192;        // 128 rows x 32 bf16
constexpr int kOutBox = 4096;       // 128 rows x 32 codes
constexpr int kBwdStages = 3;
constexpr int kBwdThreads = 32 * 9;

__host__ __device__ constexpr int bwd_stage_bytes(int d_qk) {
  return (2 * d_qk > 128 ? 2 * d_qk : 128) / 32 * kInBox;   // max(dq+q, dv) boxes
}
__host__ __device__ constexpr int bwd_smem_bytes(int d_qk, bool quant) {
  return 1024 + kBwdStages * bwd_stage_bytes(d_qk) + (quant ? 2 * 4 * kOutBox : 0);
}

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

// 16 consecutive bf16 values of row r starting at column c0 (c0 % 16 == 0)
// of a group of 32-column boxes with 64-byte swizzling.
__device__ __forceinline__ void load16(const uint8_t* boxes, int r, int c0, float (&v)[16]) {
  const uint8_t* box = boxes + (c0 >> 5) * kInBox + r * 64;
  const int cc = (c0 & 31) >> 3;
  const uint4 x0 = *reinterpret_cast<const uint4*>(box + ((cc ^ ((r >> 1) & 3)) << 4));
  const uint4 x1 = *reinterpret_cast<const uint4*>(box + (((cc + 1) ^ ((r >> 1) & 3)) << 4));
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

// mean(g_out * o) over row r of a q/k unit.
template <int DQK>
__device__ __forceinline__ float row_mean_dot(const uint8_t* in0, const uint8_t* in1, int r) {
  float dot = 0.f;
#pragma unroll 2
  for (int c0 = 0; c0 < DQK; c0 += 16) {
    float g[16], o[16];
    load16(in0, r, c0, g);
    load16(in1, r, c0, o);
#pragma unroll
    for (int j = 0; j < 16; ++j) dot = fmaf(g[j], o[j], dot);
  }
  return __fdiv_rn(dot, static_cast<float>(DQK));
}

// dY of row r of a q or k unit for 16 rotation pairs: columns [16g, 16g+16)
// into a[] and [HALF+16g, HALF+16g+16) into b[].
template <int DQK>
__device__ __forceinline__ void dy_group(const uint8_t* in0, const uint8_t* in1, int r, float mu, float rstd,
                                         const float2 (&cs)[DQK / 2], int g, float (&a)[16], float (&b)[16]) {
  constexpr int HALF = DQK / 2;
  float ga[16], gb[16], oa[16], ob[16];
  load16(in0, r, g * 16, ga);
  load16(in0, r, HALF + g * 16, gb);
  load16(in1, r, g * 16, oa);
  load16(in1, r, HALF + g * 16, ob);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float ua = ga[j] - mu * oa[j];
    const float ub = gb[j] - mu * ob[j];
    const float2 c = cs[g * 16 + j];
    a[j] = rstd * (ua * c.x + ub * c.y);
    b[j] = rstd * (ub * c.x - ua * c.y);
  }
}

// Codes of 16 consecutive columns [c0, c0+16) of row r into the token-major
// staging boxes [128 rows][32 codes].
__device__ __forceinline__ void emit16(const float (&v)[16], const Bracket& k, int r, int c0, uint8_t* out8) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = quant4_fast(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], k);
  *reinterpret_cast<uint4*>(out8 + (c0 >> 5) * kOutBox + r * 32 + (c0 & 31)) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Per-row saved state of a q/k unit: rstd and position (checked).
__device__ __forceinline__ void row_state(const BwdParams& p, const BwdUnit& b, int t, float& rstd, int& pos,
                                          const DevStatus& st, int kid) {
  rstd = 0.f;
  pos = 0;
  if (t >= p.T) return;
  rstd = __ldg(p.rstd + (static_cast<int64_t>(b.part) * p.H + b.h) * p.T + t);
  pos = __ldg(p.pos + t);
  if (pos < 0 || pos >= p.max_pos) {
    record_error(st, QKVP_ERR_DEVICE_INPUT, kid);
    pos = 0;
  }
}

__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}

// AND of `v` over the 128 threads of consumer group g (all of them call it),
// so that the group leaves its loop together.
__device__ __forceinline__ bool group_all(int g, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(v)), "r"(1 + g)
      : "memory");
  return out != 0;
}

// One kernel body for both passes.  QUANT = false: amax partials; true: codes.
template <int DQK, bool QUANT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_epi_kernel(const __grid_constant__ BwdMaps m, const __grid_constant__ BwdParams p, DevStatus st) {
  constexpr int kid = QUANT ? KID_BWD_QUANT : KID_BWD_AMAX;
  constexpr int kStage = bwd_stage_bytes(DQK);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kBwdStages], empty[kBwdStages];
  __shared__ float red[32];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 128);
    }
    fence_mbar_init();
  }
  __syncthreads();

  Bracket kq{1.f, 1.f, 1.f};
  if (QUANT) {
    const float s_dy = scale_from_amax(block_reduce_partials(p.partials, p.nparts, red));
    kq = make_bracket(s_dy);
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.dy_scale = s_dy;
  }

  float mx = 0.f;
  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      uint32_t used = 0, last_par = 0;  // stages filled; parity of their last fill
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
        const int s = it % kBwdStages;
        if (!mbar_wait(&empty[s], ((it / kBwdStages) & 1) ^ 1, &abort_flag, st, kid)) break;
        used |= 1u << s;
        last_par = (last_par & ~(1u << s)) | (static_cast<uint32_t>((it / kBwdStages) & 1) << s);
        const BwdUnit b = bwd_decode(p, u);
        uint8_t* in0 = smem + s * kStage;
        const int d = b.part < 2 ? DQK : p.d_v;
        const int nbox = d / 32;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>((b.part < 2 ? 2 : 1) * nbox * kInBox));
        const CUtensorMap* gm = b.part == 0 ? &m.dq : b.part == 1 ? &m.dk : &m.dv;
        for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + j * kInBox, gm, &full[s], 32 * j, b.t0, b.h);
        if (b.part < 2) {
          const CUtensorMap* om = b.part == 0 ? &m.q : &m.k;
          for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + (nbox + j) * kInBox, om, &full[s], 32 * j, b.t0, b.h);
        }
      }
      // every copy issued has landed before the CTA may exit
      for (int s = 0; s < kBwdStages; ++s)
        if (used & (1u << s)) mbar_wait(&full[s], (last_par >> s) & 1, nullptr, st, kid);
    }
  } else {
    const int g = (warp - 1) >> 2;                 // consumer group
    const int r = ((warp - 1) & 3) * 32 + lane;    // token row of the unit
    uint8_t* out8 = smem + kBwdStages * kStage + g * 4 * kOutBox;
    const float2* rope = reinterpret_cast<const float2*>(p.rope);
    int it = g;
    for (int u = blockIdx.x + g * gridDim.x; u < p.num_units; u += 2 * gridDim.x, it += 2) {
      const int s = it % kBwdStages;
      const BwdUnit b = bwd_decode(p, u);
      const int t = b.t0 + r;
      const bool valid = t < p.T;
      float rstd;
      int pos;
      float2 cs[DQK / 2];  // this row's cos/sin, loaded before the inputs arrive
      if (b.part < 2) {
        row_state(p, b, t, rstd, pos, st, kid);
        const float2* rope_row = rope + pos;
#pragma unroll
        for (int i = 0; i < DQK / 2; ++i) cs[i] = __ldg(rope_row + static_cast<int64_t>(i) * p.max_pos);
      }
      if (QUANT) {
        // the previous unit's stores have read this group's staging tiles
        if (r == 0) bulk_wait_read<0>();
        group_sync(g);
      }
      if (!group_all(g, mbar_wait(&full[s], (it / kBwdStages) & 1, &abort_flag, st, kid))) break;
      const uint8_t* in0 = smem + s * kStage;
      int nbox;
      if (b.part < 2) {
        const uint8_t* in1 = in0 + (DQK / 32) * kInBox;
        const float mu = row_mean_dot<DQK>(in0, in1, r);
#pragma unroll
        for (int gg = 0; gg < DQK / 32; ++gg) {
          float a[16], c[16];
          dy_group<DQK>(in0, in1, r, mu, rstd, cs, gg, a, c);
          if (!valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) a[j] = c[j] = 0.f;
          }
          if (QUANT) {
            emit16(a, kq, r, gg * 16, out8);
            emit16(c, kq, r, DQK / 2 + gg * 16, out8);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) mx = fmaxf(mx, fmaxf(fabsf(a[j]), fabsf(c[j])));
          }
        }
        nbox = DQK / 32;
      } else {
#pragma unroll 2
        for (int c0 = 0; c0 < 128; c0 += 16) {
          float v[16];
          load16(in0, r, c0, v);
          if (!valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
          }
          if (QUANT) {
            emit16(v, kq, r, c0, out8);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) mx = fmaxf(mx, fabsf(v[j]));
          }
        }
        nbox = 4;
      }
      mbar_arrive(&empty[s]);  // this thread is done with the stage
      if (QUANT) {
        fence_async_smem();
        group_sync(g);
        if (r == 0) {
          for (int j = 0; j < nbox; ++j) tma_store_2d(&m.dy8, out8 + j * kOutBox, b.col0 + 32 * j, b.t0);
          bulk_commit();
        }
      }
    }
    if (QUANT && r == 0) bulk_wait_all<0>();
  }
  if (!QUANT) {
    mx = block_max(mx, red);
    if (threadIdx.x == 0) p.partials[blockIdx.x] = mx;
  }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <int DQK, bool QUANT>
static cudaError_t launch_t(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  static bool done[64] = {};
  const int smem = bwd_smem_bytes(DQK, QUANT);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !done[dev]) {
    e = cudaFuncSetAttribute(bwd_epi_kernel<DQK, QUANT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) done[dev] = true;
  }
  bwd_epi_kernel<DQK, QUANT><<<grid, kBwdThreads, smem, s>>>(m, p, st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_amax(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  switch (p.d_qk) {
    case 64: return launch_t<64, false>(m, p, grid, st, s);
    case 96: return launch_t<96, false>(m, p, grid, st, s);
    case 128: return launch_t<128, false>(m, p, grid, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_quant(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s) {
  switch (p.d_qk) {
    case 64: return launch_t<64, true>(m, p, grid, st, s);
    case 96: return launch_t<96, true>(m, p, grid, st, s);
    case 128: return launch_t<128, true>(m, p, grid, st, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qkvp

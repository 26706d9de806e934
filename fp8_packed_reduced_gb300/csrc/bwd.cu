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
//   warp 0       TMA producer: the unit's input boxes ([128 tokens x 32 cols],
//                64-byte swizzle) into a ring of kBwdStages stages
//   warps 1-16   two consumer groups of eight warps; group g takes every
//                other unit of the CTA.  Two threads per token row: thread
//                half h owns the 8-column blocks (c / 8) % 2 == h of the row,
//                which keeps each rotation pair (i, i + d/2) in one thread;
//                the row's mean(g_out * o) is one shuffle between the two.
//                Pass 2 stages the codes of its unit (32-byte swizzle) and
//                stores them by TMA while the other group computes.
// Within a warp, lanes map to rows so that the 16-byte reads of a quarter
// warp hit eight distinct 16-byte bank groups of the swizzled boxes.
#include "kernels.cuh"

namespace qkvp {

constexpr int kInBox = 8192;        // 128 rows x 32 bf16
constexpr int kOutBox = 4096;       // 128 rows x 32 codes
constexpr int kGroupThreads = 256;
constexpr int kBwdThreads = 32 + 2 * kGroupThreads;

__host__ __device__ constexpr int bwd_stage_bytes(int d_qk) {
  return (2 * d_qk > 128 ? 2 * d_qk : 128) / 32 * kInBox;   // max(dq+q, dv) boxes
}
// As many stages as fit beside the code staging: 4 at d_qk <= 96, 3 at 128.
__host__ __device__ constexpr int bwd_stages(int d_qk) { return d_qk <= 96 ? 4 : 3; }
__host__ __device__ constexpr int bwd_smem_bytes(int d_qk, bool quant) {
  return 1024 + bwd_stages(d_qk) * bwd_stage_bytes(d_qk) + (quant ? 2 * 4 * kOutBox : 0);
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

// Row of the unit and column half owned by a consumer thread (index 0..255
// inside its group).  Lanes 8k..8k+7 of a warp cover rows {b, b+1, b+4, b+5}
// of the warp's 16 rows, both halves each.
__device__ __forceinline__ void row_and_half(int gt, int& r, int& h) {
  const int warp = gt >> 5, lane = gt & 31;
  const int j = (lane >> 1) & 3, q = lane >> 3;
  h = lane & 1;
  r = warp * 16 + (q & 1) * 2 + (q >> 1) * 8 + (j & 1) + (j >> 1) * 4;
}

// The 16-byte chunk holding columns [c, c + 8) (c % 8 == 0) of row r of a
// group of 32-column boxes with 64-byte swizzling.
__device__ __forceinline__ uint4 load8(const uint8_t* boxes, int r, int c) {
  const int cc = (c & 31) >> 3;
  return *reinterpret_cast<const uint4*>(boxes + (c >> 5) * kInBox + r * 64 + ((cc ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void unpack8(uint4 x, float (&v)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b) {
  float x[8], y[8];
  unpack8(a, x);
  unpack8(b, y);
  float d = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) d = fmaf(x[i], y[i], d);
  return d;
}

// Eight codes of columns [c, c + 8) (c % 8 == 0) of row r into the
// token-major staging boxes [128 rows][32 codes] with 32-byte swizzling
// (the 16-byte half of a row is XORed with bit 2 of the row).
__device__ __forceinline__ void emit8(const float (&v)[8], const Bracket& k, int r, int c, uint8_t* out8) {
  const uint2 w = make_uint2(quant4_fast(v[0], v[1], v[2], v[3], k), quant4_fast(v[4], v[5], v[6], v[7], k));
  const int cl = c & 31;
  *reinterpret_cast<uint2*>(out8 + (c >> 5) * kOutBox + r * 32 + (((cl >> 4) ^ ((r >> 2) & 1)) << 4) + (cl & 15)) = w;
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
  asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "n"(kGroupThreads) : "memory");
}

// AND of `v` over the threads of consumer group g (all of them call it), so
// that the group leaves its loop together.
__device__ __forceinline__ bool group_all(int g, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(v)), "r"(1 + g), "n"(kGroupThreads)
      : "memory");
  return out != 0;
}

// One kernel body for both passes.  QUANT = false: amax partials; true: codes.
template <int DQK, bool QUANT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_epi_kernel(const __grid_constant__ BwdMaps m, const __grid_constant__ BwdParams p, DevStatus st) {
  constexpr int kid = QUANT ? KID_BWD_QUANT : KID_BWD_AMAX;
  constexpr int kStage = bwd_stage_bytes(DQK);
  constexpr int kBwdStages = bwd_stages(DQK);
  constexpr int HALF = DQK / 2;      // rotation pairs per row
  constexpr int NG = HALF / 16;      // 16-pair groups; this thread owns 8 pairs of each
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[4], empty[4];
  __shared__ float red[32];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGroupThreads);
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
    const int g = (warp - 1) >> 3;                            // consumer group
    const int gt = threadIdx.x - 32 - g * kGroupThreads;      // thread index inside the group
    int r, hf;
    row_and_half(gt, r, hf);
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
      if (b.part < 2) row_state(p, b, t, rstd, pos, st, kid);
      if (QUANT) {
        // the previous unit's stores have read this group's staging tiles
        if (gt == 0) bulk_wait_read<0>();
        group_sync(g);
      }
      if (!group_all(g, mbar_wait(&full[s], (it / kBwdStages) & 1, &abort_flag, st, kid))) break;
      const uint8_t* in0 = smem + s * kStage;
      int nbox;
      if (b.part < 2) {
        const uint8_t* in1 = in0 + (DQK / 32) * kInBox;
        const float2* rope_row = rope + pos;
        float dot = 0.f;
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
          const int c = 16 * gg + 8 * hf;
          dot += dot8(load8(in0, r, c), load8(in1, r, c)) + dot8(load8(in0, r, HALF + c), load8(in1, r, HALF + c));
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);   // the row's other half
        const float mu = __fdiv_rn(dot, static_cast<float>(DQK));
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
          const int c = 16 * gg + 8 * hf;
          float2 k2[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) k2[j] = __ldg(rope_row + static_cast<int64_t>(c + j) * p.max_pos);
          float ga[8], gb[8], oa[8], ob[8], a[8], c2[8];
          unpack8(load8(in0, r, c), ga);
          unpack8(load8(in0, r, HALF + c), gb);
          unpack8(load8(in1, r, c), oa);
          unpack8(load8(in1, r, HALF + c), ob);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float ua = ga[j] - mu * oa[j];
            const float ub = gb[j] - mu * ob[j];
            a[j] = valid ? rstd * (ua * k2[j].x + ub * k2[j].y) : 0.f;
            c2[j] = valid ? rstd * (ub * k2[j].x - ua * k2[j].y) : 0.f;
          }
          if (QUANT) {
            emit8(a, kq, r, c, out8);
            emit8(c2, kq, r, HALF + c, out8);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(fabsf(a[j]), fabsf(c2[j])));
          }
        }
        mbar_arrive(&empty[s]);  // this thread is done with the stage
        nbox = DQK / 32;
      } else {
        uint4 x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = load8(in0, r, 16 * q + 8 * hf);
        mbar_arrive(&empty[s]);  // inputs now in registers
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float v[8];
          unpack8(x[q], v);
          if (!valid) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.f;
          }
          if (QUANT) {
            emit8(v, kq, r, 16 * q + 8 * hf, out8);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(v[j]));
          }
        }
        nbox = 4;
      }
      if (QUANT) {
        fence_async_smem();
        group_sync(g);
        if (gt == 0) {
          for (int j = 0; j < nbox; ++j) tma_store_2d(&m.dy8, out8 + j * kOutBox, b.col0 + 32 * j, b.t0);
          bulk_commit();
        }
      }
    }
    if (QUANT && gt == 0) bulk_wait_all<0>();
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

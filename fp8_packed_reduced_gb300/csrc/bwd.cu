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
// Work unit: 64 tokens x one head x one part (q, k or v); a group takes the
// three parts of one (token tile, head) in a row, so that the k part reuses
// the RoPE factors of the q part.  Persistent CTA per SM of four groups of
// four warps; each group owns its own ring of input stages, which one of its threads refills
// by TMA (the unit's [64 tokens x 32 cols] boxes, 64-byte swizzle) as soon
// as the group has read a stage.  Two threads per token row: thread half h
// owns the 8-column blocks (c / 8) % 2 == h of the row, which keeps each
// rotation pair (i, i + d/2) in one thread; pass 1 forms the row's
// mean(g_out * o) with one shuffle between the two and stores it in the
// workspace, and pass 2 reads it back instead of forming it again (the same
// value, so the same dY).  A thread's RoPE factors for a unit are loaded
// before its stage is awaited, and the saved rstd, position (and in pass 2
// mean) one unit ahead.  Pass 2 stages the codes of its unit (32-byte
// swizzle) and stores them by TMA while the other group computes.
// Within a warp, lanes map to rows so that the 16-byte reads of a quarter
// warp hit eight distinct 16-byte bank groups of the swizzled boxes.  In
// pass 1 the group's threads meet only through mbarriers (a stage landed;
// all have read a stage), so its warps may run apart by up to the ring's
// depth; pass 2 also meets at a group barrier per unit, before its single
// code staging is rewritten.
#include <atomic>

#include "kernels.cuh"

namespace qkvp {

constexpr int kRows = kBwdUnitRows;   // tokens per unit
constexpr int kInBox = kRows * 64;    // kRows rows x 32 bf16
constexpr int kOutBox = kRows * 32;   // kRows rows x 32 codes
constexpr int kGroupThreads = 2 * kRows;   // two threads per token row
constexpr int kGroups = 4;                 // consumer groups per CTA
constexpr int kBwdThreads = kGroups * kGroupThreads;
constexpr int kMaxStagesPerGroup = 3;

__host__ __device__ constexpr int bwd_stage_bytes(int d_qk) {
  return (2 * d_qk > 128 ? 2 * d_qk : 128) / 32 * kInBox;   // max(dq+q, dv) boxes
}
// Input stages owned by each consumer group, as many as fit beside the code
// staging: 3 at d_qk = 64 (16 KB stages), 2 at 96 (24 KB), 1 at 128 (32 KB).
__host__ __device__ constexpr int bwd_stages_per_group(int d_qk) { return d_qk <= 64 ? 3 : d_qk <= 96 ? 2 : 1; }
__host__ __device__ constexpr int bwd_smem_bytes(int d_qk, bool quant) {
  return 1024 + kGroups * bwd_stages_per_group(d_qk) * bwd_stage_bytes(d_qk) + (quant ? kGroups * 4 * kOutBox : 0);
}

struct BwdUnit {
  int part, h, t0, col0;
};

__device__ __forceinline__ BwdUnit bwd_decode(const BwdParams& p, int u) {
  BwdUnit b;
  b.part = u % 3;
  b.h = (u / 3) % p.H;
  b.t0 = (u / (3 * p.H)) * kRows;
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


// acc + the products of the eight bf16 of a with those of b, on two lanes
__device__ __forceinline__ f2 dot8(uint4 a, uint4 b, f2 acc) {
  acc = f2_fma(f2_from_bf16x2(a.x), f2_from_bf16x2(b.x), acc);
  acc = f2_fma(f2_from_bf16x2(a.y), f2_from_bf16x2(b.y), acc);
  acc = f2_fma(f2_from_bf16x2(a.z), f2_from_bf16x2(b.z), acc);
  return f2_fma(f2_from_bf16x2(a.w), f2_from_bf16x2(b.w), acc);
}

// per-half unsigned 16-bit max
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight codes of columns [c, c + 8) (c % 8 == 0) of row r into the
// token-major staging boxes [64 rows][32 codes] with 32-byte swizzling
// (the 16-byte half of a row is XORed with bit 2 of the row).
__device__ __forceinline__ void emit8(const f2 (&v)[4], const Bracket2& k, int r, int c, uint8_t* out8) {
  const uint2 w = quant8(v, k);
  const int cl = c & 31;
  *reinterpret_cast<uint2*>(out8 + (c >> 5) * kOutBox + r * 32 + (((cl >> 4) ^ ((r >> 2) & 1)) << 4) + (cl & 15)) = w;
}

// Issue the loads of a q/k unit's per-row saved state: rstd and position,
// and in pass 2 the row's mean that pass 1 stored (0 for rows past T; the
// position is range-checked where it is used).
template <bool QUANT>
__device__ __forceinline__ void row_state(const BwdParams& p, const BwdUnit& b, int t, float& rstd, int& pos,
                                          float& mu) {
  rstd = 0.f;
  pos = 0;
  mu = 0.f;
  if (t >= p.T) return;
  const int64_t row = (static_cast<int64_t>(b.part) * p.H + b.h) * p.T + t;
  rstd = __ldg(p.rstd + row);
  pos = __ldg(p.pos + t);
  if (QUANT) mu = __ldg(p.mu + row);
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

// Pass 1 keeps each q/k row's mean for pass 2: the means of four
// consecutive rows meet in lanes 0, 4, 16 and 20 (rows 0-3, 4-7, 8-11, 12-15
// of the warp) and leave as one 16-byte store where the row block is aligned
// and inside T.  Called by every lane of the warp.
__device__ __forceinline__ void store_row_means(const BwdParams& p, const BwdUnit& b, int r, float mu) {
  const float m1 = __shfl_down_sync(0xffffffffu, mu, 2);
  const float m2 = __shfl_down_sync(0xffffffffu, mu, 8);
  const float m3 = __shfl_down_sync(0xffffffffu, mu, 10);
  if ((threadIdx.x & 11) == 0) {
    const int t = b.t0 + r;
    const int64_t at = (static_cast<int64_t>(b.part) * p.H + b.h) * p.T + t;
    float* dst = p.mu + at;
    if (t + 3 < p.T && (at & 3) == 0) {
      *reinterpret_cast<float4*>(dst) = make_float4(mu, m1, m2, m3);
    } else {
      if (t < p.T) dst[0] = mu;
      if (t + 1 < p.T) dst[1] = m1;
      if (t + 2 < p.T) dst[2] = m2;
      if (t + 3 < p.T) dst[3] = m3;
    }
  }
}

// One kernel body for both passes.  QUANT = false: amax partials; true: codes.
template <int DQK, bool QUANT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_epi_kernel(const __grid_constant__ BwdMaps m, const __grid_constant__ BwdParams p, DevStatus st) {
  constexpr int kid = QUANT ? KID_BWD_QUANT : KID_BWD_AMAX;
  constexpr int kStage = bwd_stage_bytes(DQK);
  constexpr int SPG = bwd_stages_per_group(DQK);
  constexpr int HALF = DQK / 2;      // rotation pairs per row
  constexpr int NG = HALF / 16;      // 16-pair groups; this thread owns 8 pairs of each
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kGroups * kMaxStagesPerGroup];
  // per group and stage: every thread of the group is done with the stage's
  // current unit (and, in pass 2, has staged its codes); the group's thread 0
  // waits on it alone.  One barrier per stage: a thread that runs ahead can
  // only arrive again on a stage after thread 0 has refilled it, which it
  // does once the earlier phase has completed.
  __shared__ __align__(8) uint64_t done[kGroups][kMaxStagesPerGroup];
  __shared__ float red[32];
  __shared__ int abort_flag;
  const int g = threadIdx.x / kGroupThreads;    // consumer group
  const int gt = threadIdx.x % kGroupThreads;   // thread index inside the group
  int r, hf;
  row_and_half(gt, r, hf);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kGroups * SPG; ++s) mbar_init(&full[s], 1);
    for (int gg = 0; gg < kGroups; ++gg)
      for (int s = 0; s < SPG; ++s) mbar_init(&done[gg][s], kGroupThreads);
    fence_mbar_init();
  }
  __syncthreads();

  Bracket2 kq{1.f, 0, 0};
  if (QUANT) {
    const float s_dy = scale_from_amax(block_reduce_partials(p.partials, p.nparts, red));
    kq = make_bracket2(s_dy);
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.dy_scale = s_dy;
  }

  uint8_t* stages = smem + g * SPG * kStage;                 // this group's input stages
  uint8_t* out8 = smem + kGroups * SPG * kStage + g * 4 * kOutBox;  // and its code staging
  uint64_t* gfull = full + g * SPG;
  const int ustep = kGroups * gridDim.x;
  // Input loads of unit u into stage s (thread gt == 0 only).  `inflight`
  // and `inpar` record the stages whose loads have not been waited for.
  uint32_t inflight = 0, inpar = 0;
  const uint64_t stream = l2_policy_evict_first();
  auto load_unit = [&](int u, int s, uint32_t par) {
    const BwdUnit b = bwd_decode(p, u);
    uint8_t* in0 = stages + s * kStage;
    const int nbox = (b.part < 2 ? DQK : p.d_v) / 32;
    mbar_arrive_expect_tx(&gfull[s], static_cast<uint32_t>((b.part < 2 ? 2 : 1) * nbox * kInBox));
    const CUtensorMap* gm = b.part == 0 ? &m.dq : b.part == 1 ? &m.dk : &m.dv;
    const CUtensorMap* om = b.part == 0 ? &m.q : &m.k;
    if (QUANT) {
      for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + j * kInBox, gm, &gfull[s], 32 * j, b.t0, b.h);
      if (b.part < 2)
        for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + (nbox + j) * kInBox, om, &gfull[s], 32 * j, b.t0, b.h);
    } else if (u / 3 < ustep) {   // pass 1's last round: kept in L2 for pass 2's first
      for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + j * kInBox, gm, &gfull[s], 32 * j, b.t0, b.h);
      if (b.part < 2)
        for (int j = 0; j < nbox; ++j) tma_load_3d(in0 + (nbox + j) * kInBox, om, &gfull[s], 32 * j, b.t0, b.h);
    } else {
      for (int j = 0; j < nbox; ++j) tma_load_3d_hint(in0 + j * kInBox, gm, &gfull[s], 32 * j, b.t0, b.h, stream);
      if (b.part < 2)
        for (int j = 0; j < nbox; ++j)
          tma_load_3d_hint(in0 + (nbox + j) * kInBox, om, &gfull[s], 32 * j, b.t0, b.h, stream);
    }
    inflight |= 1u << s;
    inpar = (inpar & ~(1u << s)) | (par << s);
  };
  // The group's k-th unit (-1 past the end): the q, k and v parts of one
  // (token tile, head) follow each other, the (tile, head) triples going
  // round-robin over the grid's groups.  The k part reuses the q part's RoPE
  // factors (same tokens, same positions).  Pass 1 walks the triples from
  // the last token tile down, starting on the q and k the forward wrote last
  // (still in L2); pass 2 walks them upwards, starting on the inputs pass 1
  // read last.
  const int g0 = blockIdx.x + g * gridDim.x;
  const int ntriples = p.num_units / 3;
  auto unit_at = [&](int k) -> int {
    const int tr = g0 + (k / 3) * ustep;
    if (tr >= ntriples) return -1;
    return 3 * (QUANT ? tr : ntriples - 1 - tr) + k % 3;
  };
  // Pass 1 streams its inputs through L2 marked evict-first (measured 5 us
  // faster at the training shape than without a hint), except its last round,
  // which pass 2 reads first: that one is loaded without a hint (2 us off
  // pass 2; two or three such rounds, or evict-last, gained no more).  Pass 2
  // loads without a hint (evict-first there was slower).
  if (gt == 0)
    for (int k = 0; k < SPG; ++k)
      if (unit_at(k) >= 0) load_unit(unit_at(k), k, 0);

  float mx = 0.f;
  const float4* rope = reinterpret_cast<const float4*>(p.rope);
  // the saved state of the group's next q/k unit is loaded one unit ahead
  float rstd_next = 0.f, mu_next = 0.f;
  int pos_next = 0;
  if (unit_at(0) >= 0) {
    const BwdUnit b0 = bwd_decode(p, unit_at(0));
    if (b0.part < 2) row_state<QUANT>(p, b0, b0.t0 + r, rstd_next, pos_next, mu_next);
  }
  // entry w of group gg: cos, cos, sin, sin of pairs c + 2w, c + 2w + 1
  float4 k4[NG][4];
  for (int k = 0;; ++k) {
    const int u = unit_at(k);
    if (u < 0) break;
    const int s = k % SPG;
    const uint32_t par = (k / SPG) & 1;
    const BwdUnit b = bwd_decode(p, u);
    const float rstd = rstd_next, mu_row = mu_next;
    int pos = pos_next;
    // the q part's RoPE factors, in flight while the stage arrives and the
    // row's mean is formed (the k part that follows uses them again)
    if (b.part == 0) {
      if (pos < 0 || pos >= p.max_pos) {
        record_error(st, QKVP_ERR_DEVICE_INPUT, kid);
        pos = 0;
      }
      const float4* rope_row = rope + pos;
#pragma unroll
      for (int gg = 0; gg < NG; ++gg)
#pragma unroll
        for (int w = 0; w < 4; ++w)
          k4[gg][w] = __ldg(rope_row + static_cast<int64_t>(8 * gg + 4 * hf + w) * p.max_pos);
    }
    const int un = unit_at(k + 1);
    if (un >= 0) {
      const BwdUnit bn = bwd_decode(p, un);
      if (bn.part < 2) row_state<QUANT>(p, bn, bn.t0 + r, rstd_next, pos_next, mu_next);
    }
    if (QUANT) {
      // pass 2: thread 0 first lets the previous unit's codes leave the
      // staging, which this unit overwrites after the group barrier (the
      // staging is single: the group meets at every unit)
      if (gt == 0) bulk_wait_read<0>();
      if (!group_all(g, mbar_wait(&gfull[s], par, &abort_flag, st, kid) && !abort_flag)) break;
    } else {
      // pass 1: each thread waits for the stage itself, so the group's warps
      // run apart by up to the ring's depth instead of meeting at every unit
      if (!mbar_wait(&gfull[s], par, &abort_flag, st, kid) || abort_flag) break;
    }
    if (gt == 0) inflight &= ~(1u << s);
    const uint8_t* in0 = stages + s * kStage;
    int nbox;
    if (b.part < 2) {
      const uint8_t* in1 = in0 + (DQK / 32) * kInBox;
      float mu = mu_row;   // pass 2: the mean pass 1 formed (the same arithmetic)
      if (!QUANT) {
        f2 acc = 0;
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
          const int c = 16 * gg + 8 * hf;
          acc = dot8(load8(in0, r, c), load8(in1, r, c), acc);
          acc = dot8(load8(in0, r, HALF + c), load8(in1, r, HALF + c), acc);
          asm volatile("" ::: "memory");   // bounds the reads in flight (registers)
        }
        const float2 a2 = f2_split(acc);
        float dot = a2.x + a2.y;
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);   // the row's other half
        mu = __fdiv_rn(dot, static_cast<float>(DQK));
        if (DQK <= 96) store_row_means(p, b, r, mu);   // pass 1 keeps the mean for pass 2
      }
      const f2 nmu = f2_make(-mu, -mu), rr = f2_make(rstd, rstd);
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) {
        const int c = 16 * gg + 8 * hf;
        const uint4 ga = load8(in0, r, c), gb = load8(in0, r, HALF + c);
        const uint4 oa = load8(in1, r, c), ob = load8(in1, r, HALF + c);
        const uint32_t gaw[4] = {ga.x, ga.y, ga.z, ga.w}, gbw[4] = {gb.x, gb.y, gb.z, gb.w};
        const uint32_t oaw[4] = {oa.x, oa.y, oa.z, oa.w}, obw[4] = {ob.x, ob.y, ob.z, ob.w};
        f2 ya[4], yb[4];   // dY of columns c + [0, 8) and HALF + c + [0, 8), two per word
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          // u = g_out - mu * o over the pair's two columns, then the inverse rotation
          const f2 ua = f2_fma(f2_from_bf16x2(oaw[w]), nmu, f2_from_bf16x2(gaw[w]));
          const f2 ub = f2_fma(f2_from_bf16x2(obw[w]), nmu, f2_from_bf16x2(gbw[w]));
          const f2 cs = f2_make(k4[gg][w].x, k4[gg][w].y), sn = f2_make(k4[gg][w].z, k4[gg][w].w);
          ya[w] = f2_mul(f2_fma(ub, sn, f2_mul(ua, cs)), rr);
          yb[w] = f2_mul(f2_sub(f2_mul(ub, cs), f2_mul(ua, sn)), rr);
        }
        if (QUANT) {
          emit8(ya, kq, r, c, out8);
          emit8(yb, kq, r, HALF + c, out8);
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w) mx = f2_absmax(f2_absmax(mx, ya[w]), yb[w]);
          // keep the next group's shared-memory reads from being hoisted
          // above this one (their registers would spill)
          asm volatile("" ::: "memory");
        }
      }
      // (d_qk = 128: after the rotation, whose registers it would crowd)
      if (!QUANT && DQK > 96) store_row_means(p, b, r, mu);
      nbox = DQK / 32;
    } else {
      uint4 x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = load8(in0, r, 16 * q + 8 * hf);
      if (QUANT) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const f2 v[4] = {f2_from_bf16x2(x[q].x), f2_from_bf16x2(x[q].y), f2_from_bf16x2(x[q].z),
                           f2_from_bf16x2(x[q].w)};
          emit8(v, kq, r, 16 * q + 8 * hf, out8);
        }
      } else {
        // |bf16| orders as its 15 magnitude bits: max over packed halves
        uint32_t m2 = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          m2 = umax16x2(m2, x[q].x & 0x7FFF7FFFu);
          m2 = umax16x2(m2, x[q].y & 0x7FFF7FFFu);
          m2 = umax16x2(m2, x[q].z & 0x7FFF7FFFu);
          m2 = umax16x2(m2, x[q].w & 0x7FFF7FFFu);
        }
        mx = fmax3(mx, bf16_lo(m2), bf16_hi(m2));
      }
      nbox = 4;
    }
    // This thread is done with the stage: its reads are performed before the
    // arrival (release), and in pass 2 its staged codes are made visible to
    // the TMA store first.  Thread 0 alone waits for the whole group, then
    // refills the stage and stores the codes.
    if (QUANT) fence_async_smem();
    mbar_arrive(&done[g][s]);
    if (gt == 0 && mbar_wait(&done[g][s], par, &abort_flag, st, kid)) {
      if (unit_at(k + SPG) >= 0) load_unit(unit_at(k + SPG), s, par ^ 1u);
      if (QUANT) {
        for (int j = 0; j < nbox; ++j) tma_store_2d(&m.dy8, out8 + j * kOutBox, b.col0 + 32 * j, b.t0);
        bulk_commit();
      }
    }
  }
  if (gt == 0) {
    if (QUANT) bulk_wait_all<0>();
    // loads still in flight after an early exit land before the CTA ends
    for (int s = 0; s < SPG; ++s)
      if (inflight & (1u << s)) mbar_wait(&gfull[s], (inpar >> s) & 1, nullptr, st, kid);
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
  static std::atomic<bool> done[64];   // per device: the shared-memory opt-in is set
  const int smem = bwd_smem_bytes(DQK, QUANT);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !done[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(bwd_epi_kernel<DQK, QUANT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) done[dev].store(true, std::memory_order_relaxed);
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

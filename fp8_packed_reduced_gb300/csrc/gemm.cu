// The three FP8 GEMMs of the packed QKV projection, on 5th-generation tensor
// cores (tcgen05, kind::f8f6f4, fp32 accumulate in TMEM):
//   forward  acc = x8 . W8^T        epilogue: de-quantise, split, per-head
//                                   RMSNorm of q/k, RoPE, head-major bf16 store
//   dX       acc = dY8 . W8         via W8T (K-major); epilogue: scale, bf16
//   dW       acc = dY8^T . x8       MN-major operands straight from dY8 and x8,
//                                   split over K (tokens); fp32 partials,
//                                   reduced in a fixed order
//
// One persistent, warp-specialised kernel body serves all three:
//   warp 0     TMA producer: A tile (128 rows x 128 B of K) and B tile
//              (ncols rows, loaded as 32-row boxes), 128-byte swizzle
//   warp 1     TMEM allocator and MMA issuer (one thread): 4 MMAs of K = 32
//              per stage, commit to the stage's "empty" barrier, and to the
//              accumulator's "full" barrier after the last stage of a unit
//   warps 2-9  epilogue, two warps per TMEM lane quarter (each owning half of
//              the unit's heads or columns), one accumulator row (token) per
//              thread; TMEM holds two 256-column accumulators so the
//              epilogue of one unit overlaps the MMAs of the next
// Every wait is bounded (see mbar_wait); on expiry the kernel records
// QKVP_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include "kernels.cuh"

namespace qkvp {

constexpr int kBM = 128;                   // accumulator rows (tokens, or bank rows for dW)
constexpr int kBK = 128;                   // K bytes per stage (E4M3: 128 elements)
constexpr int kAStage = kBM * kBK;         // 16 KB
constexpr int kBStage = 256 * kBK;         // 32 KB (largest B tile)
// Threads of a GEMM CTA with EW epilogue warps (4 or 8).
__host__ __device__ constexpr int gemm_threads(int ew) { return 64 + 32 * ew; }
constexpr int kTmemCols = 512;             // 2 accumulators x 256 fp32 columns
constexpr int kMaxStages = 6;

struct Unit {
  int a_row, b_row, ncols, kb0, kb1;
  int b_bytes;   // bytes the B loads of one stage deliver (>= ncols * 128)
  int b_sel;     // which B tensor map the schedule loads from (forward: 0 q/k, 1 v)
};

struct GemmSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Dynamic shared memory: alignment slack, the stage ring, and `epb` bytes of
// output staging per epilogue warp (boxes of 32 rows x 64 B).
__host__ __device__ constexpr int gemm_smem_bytes(int stages, int ew, int epb) {
  return 1024 + stages * (kAStage + kBStage) + ew * epb;
}

// ---------------------------------------------------------------------------
// Producer and MMA roles (one thread each)
// ---------------------------------------------------------------------------
template <class Sched>
__device__ void producer_role(const Sched& sc, const CUtensorMap* tmA, const CUtensorMap* tmB, uint8_t* sA,
                              uint8_t* sB, GemmSmem& g, int stages, const DevStatus& st, int kid) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t used = 0, last_par = 0;  // stages filled at least once; parity of their last fill
  for (int u = blockIdx.x; u < sc.num_units(); u += gridDim.x) {
    const Unit ui = sc.unit(u);
    for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
      if (!mbar_wait(&g.empty[stage], phase ^ 1, &g.abort_flag, st, kid)) goto drain;
      mbar_arrive_expect_tx(&g.full[stage], static_cast<uint32_t>(kAStage + ui.b_bytes));
      sc.load(ui, kb, tmA, tmB, sA + stage * kAStage, sB + stage * kBStage, &g.full[stage]);
      used |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == stages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
drain:
  // every copy this thread issued has landed before the CTA may exit
  for (int s = 0; s < stages; ++s)
    if (used & (1u << s)) mbar_wait(&g.full[s], (last_par >> s) & 1, nullptr, st, kid);
}

template <class Sched>
__device__ void mma_role(const Sched& sc, uint8_t* sA, uint8_t* sB, GemmSmem& g, uint32_t tmem_base, int stages,
                         const DevStatus& st, int kid) {
  int stage = 0;
  uint32_t phase = 0;
  int it = 0;
  for (int u = blockIdx.x; u < sc.num_units(); u += gridDim.x, ++it) {
    const Unit ui = sc.unit(u);
    const int buf = it & 1;
    const uint32_t use = (it >> 1) & 1;
    if (!mbar_wait(&g.tempty[buf], use ^ 1, &g.abort_flag, st, kid)) break;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + buf * 256;
    const uint32_t idesc = idesc_e4m3_f32_major(kBM, ui.ncols, Sched::kMN, Sched::kMN);
    bool ok = true;
    for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
      if (!mbar_wait(&g.full[stage], phase, &g.abort_flag, st, kid)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + stage * kAStage), b0 = smem_u32(sB + stage * kBStage);
#pragma unroll
      for (int kk = 0; kk < kBK / 32; ++kk) {
        // K = 32 per instruction: 32 bytes along a K-major row, or 32 rows
        // (four 8-row atoms) of an MN-major tile
        const uint64_t ad = Sched::kMN ? sdesc_sw128(a0 + kk * 4096, 16384, 1024) : sdesc_k_sw128(a0 + kk * 32);
        const uint64_t bd = Sched::kMN ? sdesc_sw128(b0 + kk * 4096, 16384, 1024) : sdesc_k_sw128(b0 + kk * 32);
        umma_e4m3(d_tmem, ad, bd, idesc, (kb > ui.kb0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&g.empty[stage]);
      if (++stage == stages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok) break;
    umma_commit(&g.tfull[buf]);
  }
  // all MMAs issued by this thread have completed before TMEM is freed
  umma_commit(&g.mma_done);
  mbar_wait(&g.mma_done, 0, nullptr, st, kid);
}

// ---------------------------------------------------------------------------
// Common body
// ---------------------------------------------------------------------------
template <int EW, int EPB, class Sched, class Epi>
__device__ __forceinline__ void gemm_body(const Sched& sc, Epi& epi, const CUtensorMap* tmA,
                                          const CUtensorMap* tmB, int stages, const DevStatus& st, int kid) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ GemmSmem g;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + stages * kAStage;
  uint8_t* sE = sB + stages * kBStage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    g.abort_flag = 0;
    for (int s = 0; s < stages; ++s) {
      mbar_init(&g.full[s], 1);
      mbar_init(&g.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&g.tfull[b], 1);
      mbar_init(&g.tempty[b], EW);   // one arrival per epilogue warp
    }
    mbar_init(&g.mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(tmA);
    prefetch_tmap(tmB);
  }
  if (warp == 1) {
    tmem_alloc(&g.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = g.tmem_base;

  if (warp == 0) {
    if (lane == 0) producer_role(sc, tmA, tmB, sA, sB, g, stages, st, kid);
  } else if (warp == 1) {
    if (lane == 0) mma_role(sc, sA, sB, g, tmem_base, stages, st, kid);
  } else {
    const int qw = warp & 3;          // TMEM lane quarter this warp may access
    const int sub = (warp - 2) >> 2;  // which share of the unit's heads / columns
    epi.begin(qw, sub, EW / 4, lane, sE + (warp - 2) * EPB);
    int it = 0;
    for (int u = blockIdx.x; u < sc.num_units(); u += gridDim.x, ++it) {
      const int buf = it & 1;
      epi.prepare(u);  // loads that do not depend on the accumulator
      if (!mbar_wait(&g.tfull[buf], (it >> 1) & 1, &g.abort_flag, st, kid)) break;
      tc_fence_after();
      epi.process(u, tmem_base + static_cast<uint32_t>(buf * 256) + (static_cast<uint32_t>(qw * 32) << 16));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&g.tempty[buf]);
    }
    epi.finish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// 16-byte chunk `col / 8` of row `row` in a staging box of 32 rows x 32
// bf16 columns (64 B rows) with 64-byte swizzling, as TMA reads it.
__device__ __forceinline__ void stage_chunk_sw64(uint8_t* box, int row, int col_in_box, uint4 v) {
  const int cc = col_in_box >> 3;
  *reinterpret_cast<uint4*>(box + row * 64 + ((cc ^ ((row >> 1) & 3)) << 4)) = v;
}

// Stage 16 consecutive bf16 columns [c0, c0+16) of one row (c0 % 16 == 0)
// into a group of consecutive 2 KB boxes.
__device__ __forceinline__ void stage16(uint8_t* boxes, int row, int c0, const uint32_t (&w)[8]) {
  uint8_t* box = boxes + (c0 >> 5) * 2048;
  stage_chunk_sw64(box, row, c0 & 31, make_uint4(w[0], w[1], w[2], w[3]));
  stage_chunk_sw64(box, row, (c0 & 31) + 8, make_uint4(w[4], w[5], w[6], w[7]));
}

// K-major operands: A is one box of 128 rows x 128 bytes of K at (k, a_row);
// B is ncols/R boxes of R rows x 128 bytes at (k, b_row + R j), R = b_rows
// (the B tensor map's box height).
__device__ __forceinline__ void load_k_major(const Unit& ui, int kb, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                             uint8_t* sA, uint8_t* sB, uint64_t* bar, int b_rows) {
  tma_load_2d(sA, tmA, bar, kb * kBK, ui.a_row);
  for (int j = 0; j < ui.ncols / b_rows; ++j)
    tma_load_2d(sB + j * b_rows * kBK, tmB, bar, kb * kBK, ui.b_row + b_rows * j);
}

// ---------------------------------------------------------------------------
// Forward: schedule and epilogue
// ---------------------------------------------------------------------------
struct FwdSched {
  static constexpr bool kMN = false;
  const FwdParams& p;
  const CUtensorMap* tmBv;   // W8 with the v tiles' box height (the q/k one is the body's B map)
  // B: one box per stage, hq*d_qk rows for q/k tiles and 2*d_v rows for v
  // tiles (a narrower last tile receives the whole box; the MMA uses ncols).
  __device__ void load(const Unit& ui, int kb, const CUtensorMap* a, const CUtensorMap* b, uint8_t* sA,
                       uint8_t* sB, uint64_t* bar) const {
    tma_load_2d(sA, a, bar, kb * kBK, ui.a_row);
    tma_load_2d(sB, ui.b_sel == 0 ? b : tmBv, bar, kb * kBK, ui.b_row);
  }
  __device__ int num_units() const { return p.num_units; }
  // kind 0 = q, 1 = k, 2 = v
  __device__ void decode(int j, int& kind, int& head0, int& nh) const {
    if (j < p.nq) {
      kind = 0;
      head0 = j * p.hq;
      nh = min(p.hq, p.H - head0);
    } else if (j < 2 * p.nq) {
      kind = 1;
      head0 = (j - p.nq) * p.hq;
      nh = min(p.hq, p.H - head0);
    } else {
      kind = 2;
      head0 = (j - 2 * p.nq) * 2;
      nh = min(2, p.H - head0);
    }
  }
  __device__ Unit unit(int u) const {
    const int m = u / p.n_tiles, j = u % p.n_tiles;
    int kind, head0, nh;
    decode(j, kind, head0, nh);
    Unit r;
    r.a_row = m * kBM;
    if (kind == 0) {
      r.b_row = head0 * p.d_qk;
      r.ncols = nh * p.d_qk;
      r.b_bytes = p.hq * p.d_qk * kBK;
      r.b_sel = 0;
    } else if (kind == 1) {
      r.b_row = p.H * p.d_qk + head0 * p.d_qk;
      r.ncols = nh * p.d_qk;
      r.b_bytes = p.hq * p.d_qk * kBK;
      r.b_sel = 0;
    } else {
      r.b_row = 2 * p.H * p.d_qk + head0 * p.d_v;
      r.ncols = nh * p.d_v;
      r.b_bytes = 2 * p.d_v * kBK;
      r.b_sel = 1;
    }
    r.kb0 = 0;
    r.kb1 = p.kblocks;
    return r;
  }
};

template <int DQK>
struct FwdEpi {
  const FwdParams& p;
  const FwdSched& sc;
  const CUtensorMap* tq;
  const CUtensorMap* tk;
  const CUtensorMap* tv;
  const DevStatus& st;
  uint8_t* stage;   // 8 KB: one head's boxes
  int qw, sub, nsub, lane;
  float sxw;
  // per unit, set by prepare() before the accumulator is ready: tile decode,
  // this thread's token and its row of the RoPE table
  int kind, head0, nh, t;
  bool valid;
  const float4* rope_row;   // entry j of this token: cos, cos, sin, sin of pairs 2j, 2j + 1

  __device__ void prepare(int u) {
    const int m = u / p.n_tiles;
    sc.decode(u % p.n_tiles, kind, head0, nh);
    t = m * kBM + qw * 32 + lane;
    valid = t < p.T;
    int pos = 0;
    if (kind < 2 && valid) {
      pos = __ldg(p.pos + t);
      if (pos < 0 || pos >= p.max_pos) {
        record_error(st, QKVP_ERR_DEVICE_INPUT, KID_FWD_GEMM);
        pos = 0;
      }
    }
    rope_row = reinterpret_cast<const float4*>(p.rope) + pos;
  }

  __device__ void begin(int qw_, int sub_, int nsub_, int lane_, uint8_t* stage_) {
    qw = qw_;
    sub = sub_;
    nsub = nsub_;
    lane = lane_;
    stage = stage_;
    sxw = (*p.x_scale) * (*p.w_scale);
  }
  __device__ void finish() {
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  }
  // wait until the previous head's store has read the staging boxes
  __device__ uint8_t* acquire() {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    return stage;
  }

  __device__ void process(int u, uint32_t tacc) {
    constexpr int HALF = DQK / 2;
    const int ty = (u / p.n_tiles) * kBM + qw * 32;
    for (int hh = sub; hh < nh; hh += nsub) {  // this warp's heads of the unit
      const int h = head0 + hh;
      uint8_t* buf = acquire();
      if (kind < 2) {
        // pass 1: sum of squares of the raw accumulators (scaled once below)
        f2 ss2 = 0;
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c) {
          uint32_t raw[32];
          tmem_ld16(tacc + hh * DQK + 32 * c, raw);
          tmem_ld16(tacc + hh * DQK + 32 * c + 16, raw + 16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const f2 v = f2_make(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
            ss2 = f2_fma(v, v, ss2);
          }
        }
        const float2 ssp = f2_split(ss2);
        const float ss = (ssp.x + ssp.y) * (sxw * sxw);
        const float r = 1.0f / sqrtf(__fdiv_rn(ss, static_cast<float>(DQK)) + p.eps);
        if (valid) p.rstd[(static_cast<int64_t>(kind) * p.H + h) * p.T + t] = r;
        const f2 f = f2_make(sxw * r, sxw * r);   // accumulator -> normalised value
        // pass 2: rotate 16 pairs at a time, columns [16g, 16g+16) and [HALF+16g, HALF+16g+16)
#pragma unroll
        for (int g = 0; g < HALF / 16; ++g) {
          float4 cs[8];
#pragma unroll
          for (int w = 0; w < 8; ++w) cs[w] = __ldg(rope_row + static_cast<int64_t>(g * 8 + w) * p.max_pos);
          uint32_t ra[16], rb[16];
          tmem_ld16(tacc + hh * DQK + g * 16, ra);
          tmem_ld16(tacc + hh * DQK + HALF + g * 16, rb);
          tmem_ld_wait();
          uint32_t lo[8], hi[8];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const f2 a = f2_mul(f2_make(__uint_as_float(ra[2 * w]), __uint_as_float(ra[2 * w + 1])), f);
            const f2 b = f2_mul(f2_make(__uint_as_float(rb[2 * w]), __uint_as_float(rb[2 * w + 1])), f);
            const f2 c = f2_make(cs[w].x, cs[w].y), sn = f2_make(cs[w].z, cs[w].w);
            lo[w] = f2_to_bf16x2(f2_sub(f2_mul(a, c), f2_mul(b, sn)));   // a cos - b sin
            hi[w] = f2_to_bf16x2(f2_fma(a, sn, f2_mul(b, c)));           // b cos + a sin
          }
          stage16(buf, lane, g * 16, lo);
          stage16(buf, lane, HALF + g * 16, hi);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const CUtensorMap* map = kind == 0 ? tq : tk;
#pragma unroll
          for (int b = 0; b < DQK / 32; ++b) tma_store_3d(map, buf + b * 2048, 32 * b, ty, h);
          bulk_commit();
        }
      } else {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t raw[64];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(tacc + hh * 128 + hf * 64 + 16 * c, raw + 16 * c);
          tmem_ld_wait();
          const f2 sc = f2_make(sxw, sxw);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = f2_to_bf16x2(
                  f2_mul(f2_make(__uint_as_float(raw[g * 16 + 2 * i]), __uint_as_float(raw[g * 16 + 2 * i + 1])), sc));
            stage16(buf, lane, hf * 64 + g * 16, w);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int b = 0; b < 4; ++b) tma_store_3d(tv, buf + b * 2048, 32 * b, ty, h);
          bulk_commit();
        }
      }
    }
  }
};

// Epilogue warps and per-warp staging bytes of each GEMM.
constexpr int kFwdEW = 8, kDxEW = 4, kDwEW = 8;
constexpr int kFwdEPB = 8192, kDxEPB = 8192;

template <int DQK>
__global__ void __launch_bounds__(gemm_threads(kFwdEW), 1)
    fwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBv,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ FwdParams p, DevStatus st,
                    int stages) {
  FwdSched sc{p, &tmBv};
  FwdEpi<DQK> epi{p, sc, &tq, &tk, &tv, st};
  gemm_body<kFwdEW, kFwdEPB>(sc, epi, &tmA, &tmB, stages, st, KID_FWD_GEMM);
}

// ---------------------------------------------------------------------------
// dX: schedule and epilogue
// ---------------------------------------------------------------------------
struct DxSched {
  static constexpr bool kMN = false;
  const DxParams& p;
  __device__ void load(const Unit& ui, int kb, const CUtensorMap* a, const CUtensorMap* b, uint8_t* sA,
                       uint8_t* sB, uint64_t* bar) const {
    load_k_major(ui, kb, a, b, sA, sB, bar, p.bn);
  }
  __device__ int num_units() const { return p.num_units; }
  __device__ Unit unit(int u) const {
    Unit r;
    r.a_row = (u / p.n_tiles) * kBM;
    r.b_row = (u % p.n_tiles) * p.bn;
    r.ncols = p.bn;
    r.b_bytes = p.bn * kBK;
    r.b_sel = 0;
    r.kb0 = 0;
    r.kb1 = p.kblocks;
    return r;
  }
};

struct DxEpi {
  const DxParams& p;
  const CUtensorMap* tdx;
  uint8_t* stage;
  int qw, sub, nsub, lane, ring;
  float sc;
  __device__ void begin(int qw_, int sub_, int nsub_, int lane_, uint8_t* stage_) {
    qw = qw_;
    sub = sub_;
    nsub = nsub_;
    lane = lane_;
    stage = stage_;
    ring = 0;
    sc = (*p.dy_scale) * (*p.w_scale);
  }
  __device__ void finish() {
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  }
  __device__ void prepare(int) {}
  __device__ void process(int u, uint32_t tacc) {
    const int m = u / p.n_tiles, j = u % p.n_tiles;
    const int ty = m * kBM + qw * 32;
    const int share = p.bn / nsub;   // this warp's columns: [sub * share, (sub + 1) * share)
    for (int c0 = sub * share; c0 < (sub + 1) * share; c0 += 32) {
      uint8_t* slot = stage + (ring & 3) * 2048;
      if (lane == 0) bulk_wait_read<3>();
      __syncwarp();
      uint32_t raw[32];
      tmem_ld16(tacc + c0, raw);
      tmem_ld16(tacc + c0 + 16, raw + 16);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = pack_bf16x2(__uint_as_float(raw[g * 16 + 2 * i]) * sc, __uint_as_float(raw[g * 16 + 2 * i + 1]) * sc);
        stage16(slot, lane, g * 16, w);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tdx, slot, j * p.bn + c0, ty);
        bulk_commit();
      }
      ++ring;
    }
  }
};

__global__ void __launch_bounds__(gemm_threads(kDxEW), 1)
    dx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tdx, const __grid_constant__ DxParams p, DevStatus st,
                   int stages) {
  DxSched sc{p};
  DxEpi epi{p, &tdx};
  gemm_body<kDxEW, kDxEPB>(sc, epi, &tmA, &tmB, stages, st, KID_DX_GEMM);
}

// ---------------------------------------------------------------------------
// dW: split-K schedule, fp32 partial epilogue, fixed-order reduction.
// dW = dY8^T . x8 reads both operands MN-major straight from the token-major
// tensors: a 128-token slice of dY8 [T, N] is the A tile (M = packed rows,
// contiguous) and of x8 [T, D] the B tile (N = model columns, contiguous).
// Token rows past T are zero-filled by TMA.
// ---------------------------------------------------------------------------
struct DwSched {
  static constexpr bool kMN = true;
  const DwParams& p;
  // A: one box of 128 tokens x 128 packed columns at (a_row, k); B: ncols/128
  // boxes of 128 tokens x 128 model columns at (b_row + 128 j, k).
  __device__ void load(const Unit& ui, int kb, const CUtensorMap* a, const CUtensorMap* b, uint8_t* sA,
                       uint8_t* sB, uint64_t* bar) const {
    tma_load_2d(sA, a, bar, ui.a_row, kb * kBK);
    for (int j = 0; j < ui.ncols / 128; ++j) tma_load_2d(sB + j * 16384, b, bar, ui.b_row + 128 * j, kb * kBK);
  }
  __device__ int num_units() const { return p.num_units; }
  __device__ Unit unit(int u) const {
    const int mn = p.m_tiles * p.n_tiles;
    const int tile = u % mn, split = u / mn;
    Unit r;
    r.a_row = (tile / p.n_tiles) * kBM;
    r.b_row = (tile % p.n_tiles) * p.bn;
    r.ncols = p.bn;
    r.b_bytes = p.bn * kBK;
    r.b_sel = 0;
    r.kb0 = static_cast<int>(static_cast<int64_t>(split) * p.kblocks_total / p.splits);
    r.kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.kblocks_total / p.splits);
    return r;
  }
};

struct DwEpi {
  const DwParams& p;
  int qw, sub, nsub, lane;
  __device__ void begin(int qw_, int sub_, int nsub_, int lane_, uint8_t*) {
    qw = qw_;
    sub = sub_;
    nsub = nsub_;
    lane = lane_;
  }
  __device__ void finish() {}
  __device__ void prepare(int) {}
  __device__ void process(int u, uint32_t tacc) {
    // unit u owns partials[u][bn][128] (column-major tile): coalesced stores
    float* dst = p.partials + static_cast<int64_t>(u) * p.bn * kBM + qw * 32 + lane;
    const int share = p.bn / nsub;
    for (int c0 = sub * share; c0 < (sub + 1) * share; c0 += 32) {
      uint32_t raw[32];
      tmem_ld16(tacc + c0, raw);
      tmem_ld16(tacc + c0 + 16, raw + 16);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[static_cast<int64_t>(c0 + i) * kBM] = __uint_as_float(raw[i]);
    }
  }
};

__global__ void __launch_bounds__(gemm_threads(kDwEW), 1)
    dw_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ DwParams p, DevStatus st, int stages) {
  DwSched sc{p};
  DwEpi epi{p};
  gemm_body<kDwEW, 0>(sc, epi, &tmA, &tmB, stages, st, KID_DW_GEMM);
}

// dW[n][d] = bf16(s_dy * s_x * sum over splits, in split order, of the
// partials).  One thread per (row, 4 columns): all of its splits' loads are
// issued before the first add.  grid: (m_tiles * n_tiles, bn / 4), 128 threads.
constexpr int kMaxReduceSplits = 16;
__global__ void __launch_bounds__(128) dw_reduce_kernel(const __grid_constant__ DwParams p, const float* dy_scale,
                                                        const float* x_scale, uint16_t* dW) {
  const int tile = blockIdx.x, c0 = blockIdx.y * 4;
  const int row = threadIdx.x;
  const int mn = p.m_tiles * p.n_tiles;
  float v[kMaxReduceSplits][4];
#pragma unroll
  for (int s = 0; s < kMaxReduceSplits; ++s)
    if (s < p.splits) {
      const float* src = p.partials + (static_cast<int64_t>(s * mn + tile) * p.bn + c0) * kBM + row;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[s][i] = __ldcs(src + i * kBM);
    }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < kMaxReduceSplits; ++s)
    if (s < p.splits)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += v[s][i];
  const int n = (tile / p.n_tiles) * kBM + row;
  if (n >= p.N) return;
  const int d = (tile % p.n_tiles) * p.bn + c0;
  const float sc = (*dy_scale) * (*x_scale);
  *reinterpret_cast<uint2*>(dW + static_cast<int64_t>(n) * p.D + d) =
      make_uint2(pack_bf16x2(acc[0] * sc, acc[1] * sc), pack_bf16x2(acc[2] * sc, acc[3] * sc));
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
constexpr int kFwdStages = 3, kDxStages = 4, kDwStages = 4;

template <class K>
static cudaError_t set_smem_once(K kernel, int bytes, bool (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) done[dev] = true;
  return e;
}

template <int DQK>
static cudaError_t launch_fwd_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBv,
                                const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p, int grid,
                                DevStatus st, cudaStream_t s) {
  static bool done[64] = {};
  const int smem = gemm_smem_bytes(kFwdStages, kFwdEW, kFwdEPB);
  cudaError_t e = set_smem_once(fwd_gemm_kernel<DQK>, smem, done);
  if (e != cudaSuccess) return e;
  fwd_gemm_kernel<DQK><<<grid, gemm_threads(kFwdEW), smem, s>>>(tmA, tmB, tmBv, tq, tk, tv, p, st, kFwdStages);
  return cudaGetLastError();
}

cudaError_t launch_fwd_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBv,
                            const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                            int grid, DevStatus st, cudaStream_t s) {
  switch (p.d_qk) {
    case 64: return launch_fwd_t<64>(tmA, tmB, tmBv, tq, tk, tv, p, grid, st, s);
    case 96: return launch_fwd_t<96>(tmA, tmB, tmBv, tq, tk, tv, p, grid, st, s);
    case 128: return launch_fwd_t<128>(tmA, tmB, tmBv, tq, tk, tv, p, grid, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dx_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tdx,
                           const DxParams& p, int grid, DevStatus st, cudaStream_t s) {
  static bool done[64] = {};
  const int smem = gemm_smem_bytes(kDxStages, kDxEW, kDxEPB);
  cudaError_t e = set_smem_once(dx_gemm_kernel, smem, done);
  if (e != cudaSuccess) return e;
  dx_gemm_kernel<<<grid, gemm_threads(kDxEW), smem, s>>>(tmA, tmB, tdx, p, st, kDxStages);
  return cudaGetLastError();
}

cudaError_t launch_dw_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const DwParams& p, int grid,
                           DevStatus st, cudaStream_t s) {
  static bool done[64] = {};
  const int smem = gemm_smem_bytes(kDwStages, kDwEW, 0);
  cudaError_t e = set_smem_once(dw_gemm_kernel, smem, done);
  if (e != cudaSuccess) return e;
  dw_gemm_kernel<<<grid, gemm_threads(kDwEW), smem, s>>>(tmA, tmB, p, st, kDwStages);
  return cudaGetLastError();
}

cudaError_t launch_dw_reduce(const DwParams& p, const float* dy_scale, const float* x_scale, uint16_t* dW,
                             cudaStream_t s) {
  if (p.splits > kMaxReduceSplits) return cudaErrorInvalidValue;
  dw_reduce_kernel<<<dim3(p.m_tiles * p.n_tiles, p.bn / 4), 128, 0, s>>>(p, dy_scale, x_scale, dW);
  return cudaGetLastError();
}

}  // namespace qkvp

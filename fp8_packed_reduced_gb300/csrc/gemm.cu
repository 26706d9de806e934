// The three FP8 GEMMs of the packed QKV projection, on 5th-generation tensor
// cores (tcgen05, kind::f8f6f4, fp32 accumulate in TMEM):
//   forward  acc = x8 . W8^T        epilogue: de-quantise, split, per-head
//                                   RMSNorm of q/k, RoPE, head-major bf16 store
//   dX       acc = dY8 . W8         via W8T (K-major); epilogue: scale, bf16
//   dW       acc = dY8^T . x8       MN-major operands straight from dY8 and x8,
//                                   split over K (tokens); fp32 partials,
//                                   summed in split order by a second kernel
//
// One persistent, warp-specialised kernel body serves all three:
//   warp 0     TMA producer: A tile (128 rows x 128 B of K) and B tile
//              (one box of the tile's rows), 128-byte swizzle
//   warp 1     TMEM allocator and MMA issuer (one thread): 4 MMAs of K = 32
//              per stage, commit to the stage's "empty" barrier, and to the
//              accumulator's "full" barrier after the last stage of a unit
//   warps 2-   epilogue, four or eight warps (one or two per TMEM lane
//              quarter, each owning a share of the unit's heads or columns),
//              one accumulator row (token) per thread; TMEM holds two
//              256-column accumulators so the epilogue of one unit overlaps
//              the MMAs of the next
// On CTA pairs (a 2-CTA cluster, cta_group::2) a unit is a 256-row tile:
// each CTA loads its own 128 rows of A and half of B (both halves complete
// on the even CTA's stage barrier), the even CTA's MMA thread issues M = 256
// MMAs over both CTAs' shared memory, each CTA's epilogue reads its own TMEM
// rows, and the MMA commits arrive on both CTAs' barriers.  Per SM this halves
// the bytes of B that TMA loads and writes into shared memory.
// Every wait is bounded (see mbar_wait); on expiry the kernel records
// QKVP_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <atomic>
#include <utility>

#include "kernels.cuh"

namespace qkvp {

constexpr int kBM = 128;                   // accumulator rows (tokens, or bank rows for dW)
constexpr int kBK = 128;                   // K bytes per stage (E4M3: 128 elements)
constexpr int kAStage = kBM * kBK;         // 16 KB
// Dynamic shared memory a GEMM CTA may use: the 227 KB opt-in limit less
// 1 KB for the static barriers.
constexpr int kSmemMax = 232448 - 1024;
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
  uint64_t full[kMaxStages];    // a stage landed (in a pair: both CTAs' halves, on the even CTA's barrier)
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// The stage ring: `stages` slots of one A tile and one B tile of up to
// `bstage` bytes (a multiple of 1024, the 128-byte swizzle atom).
struct Ring {
  int stages, bstage;
};

// Dynamic shared memory: alignment slack, the stage ring, and `epb` bytes of
// output staging per epilogue warp (boxes of 32 rows).
__host__ __device__ constexpr int gemm_smem_bytes(Ring r, int ew, int epb) {
  return 1024 + r.stages * (kAStage + r.bstage) + ew * epb;
}
// As many stages of (A, `bstage`-byte B) as fit beside the staging.
__host__ __device__ constexpr Ring ring_for(int bstage, int ew, int epb) {
  return Ring{(kSmemMax - 1024 - ew * epb) / (kAStage + bstage) < kMaxStages
                  ? (kSmemMax - 1024 - ew * epb) / (kAStage + bstage)
                  : kMaxStages,
              bstage};
}

// Units are distributed over CTAs, or over CTA pairs (2-CTA clusters, ranks
// 0 and 1 at consecutive block indices) that compute one 256-row tile.
template <bool PAIR>
__device__ __forceinline__ int unit_first() {
  return PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
}
template <bool PAIR>
__device__ __forceinline__ int unit_stride() {
  return PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
}

// ---------------------------------------------------------------------------
// Producer and MMA roles (one thread each)
// ---------------------------------------------------------------------------
// Loads this CTA's operand tiles (its A rows and, in a pair, its half of B).
// In a pair both CTAs' copies of a stage complete on the even CTA's `full`
// barrier, which the even CTA arms with the bytes of both halves (a copy of
// the odd CTA may land before that arming: the phase cannot complete while
// the arrival is missing).
template <bool PAIR, class Sched>
__device__ void producer_role(const Sched& sc, const CUtensorMap* tmA, const CUtensorMap* tmB, uint8_t* sA,
                              uint8_t* sB, GemmSmem& g, Ring ring, const DevStatus& st, int kid) {
  const int stages = ring.stages;
  const bool leader = !PAIR || cluster_rank() == 0;
  const uint32_t full0 = PAIR ? mapa_rank(&g.full[0], 0) : smem_u32(&g.full[0]);
  int stage = 0;
  uint32_t phase = 0;
  uint32_t used = 0, last_par = 0;  // stages filled at least once; parity of their last fill
  bool aborted = false;
  for (int u = unit_first<PAIR>(); u < sc.num_units(); u += unit_stride<PAIR>()) {
    const Unit ui = sc.unit(u);
    for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
      if (!mbar_wait(&g.empty[stage], phase ^ 1, &g.abort_flag, st, kid)) {
        aborted = true;
        goto drain;
      }
      if (leader) mbar_arrive_expect_tx(&g.full[stage], static_cast<uint32_t>((PAIR ? 2 : 1) * (kAStage + ui.b_bytes)));
      sc.template load<PAIR>(ui, kb, tmA, tmB, sA + stage * kAStage, sB + stage * ring.bstage,
                             full0 + 8u * static_cast<uint32_t>(stage));
      used |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == stages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
drain:
  // every copy issued here has landed before the CTA may exit
  if (leader) {
    for (int s = 0; s < stages; ++s)
      if (used & (1u << s)) mbar_wait(&g.full[s], (last_par >> s) & 1, nullptr, st, kid);
  } else if (aborted) {
    // The odd CTA cannot observe the even CTA's barrier: after an abort it
    // waits 100 us, far longer than any copy from device memory takes.  (On
    // the normal path the even CTA's MMAs consume every copy before the
    // pair's final cluster barrier.)
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
}

// Issues the MMAs (the even CTA of a pair issues them for both CTAs, M = 256).
template <bool PAIR, class Sched>
__device__ void mma_role(const Sched& sc, uint8_t* sA, uint8_t* sB, GemmSmem& g, uint32_t tmem_base, Ring ring,
                         const DevStatus& st, int kid) {
  const int stages = ring.stages;
  int stage = 0;
  uint32_t phase = 0;
  int it = 0;
  for (int u = unit_first<PAIR>(); u < sc.num_units(); u += unit_stride<PAIR>(), ++it) {
    const Unit ui = sc.unit(u);
    const int buf = it & 1;
    const uint32_t use = (it >> 1) & 1;
    // both CTAs' epilogues have read this accumulator buffer
    if (!(PAIR ? mbar_wait_cl(&g.tempty[buf], use ^ 1, &g.abort_flag, st, kid)
               : mbar_wait(&g.tempty[buf], use ^ 1, &g.abort_flag, st, kid)))
      break;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + buf * 256;
    const uint32_t idesc = idesc_e4m3_f32_major(PAIR ? 2 * kBM : kBM, ui.ncols, Sched::kMN, Sched::kMN);
    bool ok = true;
    for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
      if (!mbar_wait(&g.full[stage], phase, &g.abort_flag, st, kid)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + stage * kAStage), b0 = smem_u32(sB + stage * ring.bstage);
#pragma unroll
      for (int kk = 0; kk < kBK / 32; ++kk) {
        // K = 32 per instruction: 32 bytes along a K-major row, or 32 rows
        // (four 8-row atoms) of an MN-major tile
        const uint64_t ad = Sched::kMN ? sdesc_sw128(a0 + kk * 4096, 16384, 1024) : sdesc_k_sw128(a0 + kk * 32);
        const uint64_t bd = Sched::kMN ? sdesc_sw128(b0 + kk * 4096, 16384, 1024) : sdesc_k_sw128(b0 + kk * 32);
        umma_e4m3_t<PAIR>(d_tmem, ad, bd, idesc, (kb > ui.kb0 || kk > 0) ? 1u : 0u);
      }
      umma_commit_t<PAIR>(&g.empty[stage]);
      if (++stage == stages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!ok) break;
    umma_commit_t<PAIR>(&g.tfull[buf]);
  }
  // all MMAs issued by this thread have completed before TMEM is freed
  umma_commit_t<PAIR>(&g.mma_done);
  mbar_wait(&g.mma_done, 0, nullptr, st, kid);
}


// ---------------------------------------------------------------------------
// Common body
// ---------------------------------------------------------------------------
template <int EW, int EPB, bool PAIR, class Sched, class Epi>
__device__ __forceinline__ void gemm_body(const Sched& sc, Epi& epi, const CUtensorMap* tmA,
                                          const CUtensorMap* tmB, Ring ring, const DevStatus& st, int kid) {
  const int stages = ring.stages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ GemmSmem g;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + stages * kAStage;
  uint8_t* sE = sB + stages * ring.bstage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool leader = !PAIR || cluster_rank() == 0;

  if (threadIdx.x == 0) {
    g.abort_flag = 0;
    for (int s = 0; s < stages; ++s) {
      mbar_init(&g.full[s], 1);
      mbar_init(&g.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&g.tfull[b], 1);
      mbar_init(&g.tempty[b], PAIR ? 2 * EW : EW);   // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(&g.mma_done, 1);
    fence_mbar_init();
    prefetch_tmap(tmA);
    prefetch_tmap(tmB);
  }
  if (warp == 1) {
    tmem_alloc_t<PAIR>(&g.tmem_base, kTmemCols);
    tmem_relinquish_t<PAIR>();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();   // the peer's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = g.tmem_base;

  if (warp == 0) {
    if (lane == 0) producer_role<PAIR>(sc, tmA, tmB, sA, sB, g, ring, st, kid);
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader)
        mma_role<PAIR>(sc, sA, sB, g, tmem_base, ring, st, kid);
      else   // the odd CTA's memory and TMEM stay in use until the pair's MMAs are done
        mbar_wait(&g.mma_done, 0, nullptr, st, kid);
    }
  } else {
    const int qw = warp & 3;          // TMEM lane quarter this warp may access
    const int sub = (warp - 2) >> 2;  // which share of the unit's heads / columns
    epi.begin(qw, sub, EW / 4, lane, sE + (warp - 2) * EPB);
    const uint32_t tempty0 = PAIR ? mapa_rank(&g.tempty[0], 0) : 0;
    int it = 0;
    for (int u = unit_first<PAIR>(); u < sc.num_units(); u += unit_stride<PAIR>(), ++it) {
      const int buf = it & 1;
      epi.prepare(u);  // loads that do not depend on the accumulator
      if (!mbar_wait(&g.tfull[buf], (it >> 1) & 1, &g.abort_flag, st, kid)) break;
      tc_fence_after();
      // The epilogue calls `release` (once, with the whole warp) as soon as
      // its last read of the accumulator has completed, so that the MMAs of
      // a later unit may overwrite the buffer while it finishes.
      bool released = false;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR)
            mbar_arrive_cluster(tempty0 + 8u * static_cast<uint32_t>(buf));
          else
            mbar_arrive(&g.tempty[buf]);
        }
        released = true;
      };
      epi.process(u, tmem_base + static_cast<uint32_t>(buf * 256) + (static_cast<uint32_t>(qw * 32) << 16), release);
      if (!released) release();
      epi.post(u);   // work after the accumulator buffer is released
    }
    epi.finish();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();   // neither CTA leaves while the other may still address it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_t<PAIR>(tmem_base, kTmemCols);
}

// 16-byte chunk `col / 8` of row `row` in a staging box of 32 rows x 32
// bf16 columns (64 B rows) with 64-byte swizzling, as TMA reads it.
__device__ __forceinline__ void stage_chunk_sw64(uint8_t* box, int row, int col_in_box, uint4 v) {
  const int cc = col_in_box >> 3;
  *reinterpret_cast<uint4*>(box + row * 64 + ((cc ^ ((row >> 1) & 3)) << 4)) = v;
}

// Stage 16 consecutive bf16 columns [c0, c0+16) of one row (c0 % 16 == 0)
// into consecutive boxes of 32 rows x 64 columns (128 B rows, 128-byte
// swizzling: the 16-byte chunk index is XORed with the row's low three bits).
__device__ __forceinline__ void stage16_sw128(uint8_t* boxes, int row, int c0, const uint32_t (&w)[8]) {
  uint8_t* box = boxes + (c0 >> 6) * 4096 + row * 128;
  const int cc = (c0 & 63) >> 3;
  *reinterpret_cast<uint4*>(box + ((cc ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(box + (((cc + 1) ^ (row & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Stage 16 consecutive bf16 columns [c0, c0+16) of one row (c0 % 16 == 0)
// into a group of consecutive 2 KB boxes.
__device__ __forceinline__ void stage16(uint8_t* boxes, int row, int c0, const uint32_t (&w)[8]) {
  uint8_t* box = boxes + (c0 >> 5) * 2048;
  stage_chunk_sw64(box, row, c0 & 31, make_uint4(w[0], w[1], w[2], w[3]));
  stage_chunk_sw64(box, row, (c0 & 31) + 8, make_uint4(w[4], w[5], w[6], w[7]));
}

// ---------------------------------------------------------------------------
// Forward: schedule and epilogue
// ---------------------------------------------------------------------------
struct FwdSched {
  static constexpr bool kMN = false;
  const FwdParams& p;
  const CUtensorMap* tmBv;   // W8 with the v tiles' box height (the q/k one is the body's B map)
  int rank, pair;            // CTA within its pair (0 when unpaired), CTAs per unit (1 or 2)
  // 128-row block of tokens this CTA computes for unit u
  __device__ int mtile(int u) const { return (u / p.n_tiles) * pair + rank; }
  // B: one box per stage, hq*d_qk rows for q/k tiles and 2*d_v rows for v
  // tiles, or in a pair this CTA's half of them (starting ncols/2 rows in for
  // the odd CTA); a narrower last tile receives the whole box, the MMA uses
  // ncols.
  template <bool PAIR>
  __device__ void load(const Unit& ui, int kb, const CUtensorMap* a, const CUtensorMap* b, uint8_t* sA,
                       uint8_t* sB, uint32_t bar) const {
    tma_load_2d_at<PAIR>(sA, a, bar, kb * kBK, ui.a_row);
    tma_load_2d_at<PAIR>(sB, ui.b_sel == 0 ? b : tmBv, bar, kb * kBK, ui.b_row);
  }
  __device__ int num_units() const { return p.num_units; }
  // tile (index into q tiles, then k tiles, then v tiles) of unit u
  __device__ int tile(int u) const { return p.tile_order[u % p.n_tiles]; }
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
    const int j = tile(u);
    int kind, head0, nh;
    decode(j, kind, head0, nh);
    Unit r;
    r.a_row = mtile(u) * kBM;
    if (kind == 0) {
      r.b_row = head0 * p.d_qk;
      r.ncols = nh * p.d_qk;
      r.b_bytes = p.hq * p.d_qk / pair * kBK;
      r.b_sel = 0;
    } else if (kind == 1) {
      r.b_row = p.H * p.d_qk + head0 * p.d_qk;
      r.ncols = nh * p.d_qk;
      r.b_bytes = p.hq * p.d_qk / pair * kBK;
      r.b_sel = 0;
    } else {
      r.b_row = 2 * p.H * p.d_qk + head0 * p.d_v;
      r.ncols = nh * p.d_v;
      r.b_bytes = 2 * p.d_v / pair * kBK;
      r.b_sel = 1;
    }
    r.b_row += rank * (r.ncols / pair);
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
  uint8_t* stage;   // 4 KB: one box of 32 rows x 64 columns
  int qw, sub, nsub, lane;
  float sxw;
  // per unit, set by prepare() before the accumulator is ready: tile decode,
  // this thread's token and its row of the RoPE table
  int kind, head0, nh, t;
  bool valid;
  const float4* rope_row;   // entry j of this token: cos, cos, sin, sin of pairs 2j, 2j + 1

  __device__ void post(int) {}
  __device__ void prepare(int u) {
    const int m = sc.mtile(u);
    sc.decode(sc.tile(u), kind, head0, nh);
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
  // wait until the previous store has read the staging box
  __device__ uint8_t* acquire() {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    return stage;
  }
  // the staged box goes to columns [x0, x0 + 64) of head h, rows ty..ty+31
  __device__ void store_box(const CUtensorMap* map, int x0, int ty, int h) {
    fence_async_smem();
    __syncwarp();
    if (lane == 0 && ty < p.T) {   // (a pair's second tile may lie wholly past T)
      tma_store_3d(map, stage, x0, ty, h);
      bulk_commit();
    }
  }

  // One head's output leaves in 64-column boxes through the warp's single
  // staging box: columns [0, 64) first, then (d > 64) columns [64, d), the
  // columns of that box past d lying outside the tensor and not written.
  template <class Release>
  __device__ void process(int u, uint32_t tacc, Release& release) {
    constexpr int HALF = DQK / 2;
    constexpr int NG = HALF / 16;                           // rotation groups of 16 pairs
    constexpr int G1 = HALF >= 64 ? 0 : (64 - HALF) / 16;   // groups whose upper columns lie in box 0
    const int ty = sc.mtile(u) * kBM + qw * 32;
    for (int hh = sub; hh < nh; hh += nsub) {  // this warp's heads of the unit
      const int h = head0 + hh;
      const bool last_head = hh + nsub >= nh;
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
        // pass 2: rotate 16 pairs at a time, columns [16g, 16g+16) and
        // [HALF+16g, HALF+16g+16); upper columns at or past 64 wait in
        // registers until box 0 has left
        uint32_t keep[NG - G1 > 0 ? NG - G1 : 1][8];
        uint8_t* buf = acquire();
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float4 cs[8];
#pragma unroll
          for (int w = 0; w < 8; ++w) cs[w] = __ldg(rope_row + static_cast<int64_t>(g * 8 + w) * p.max_pos);
          uint32_t ra[16], rb[16];
          tmem_ld16(tacc + hh * DQK + g * 16, ra);
          tmem_ld16(tacc + hh * DQK + HALF + g * 16, rb);
          tmem_ld_wait();
          if (last_head && g == NG - 1) release();
          uint32_t lo[8], hi[8];
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const f2 a = f2_mul(f2_make(__uint_as_float(ra[2 * w]), __uint_as_float(ra[2 * w + 1])), f);
            const f2 b = f2_mul(f2_make(__uint_as_float(rb[2 * w]), __uint_as_float(rb[2 * w + 1])), f);
            const f2 c = f2_make(cs[w].x, cs[w].y), sn = f2_make(cs[w].z, cs[w].w);
            lo[w] = f2_to_bf16x2(f2_sub(f2_mul(a, c), f2_mul(b, sn)));   // a cos - b sin
            hi[w] = f2_to_bf16x2(f2_fma(a, sn, f2_mul(b, c)));           // b cos + a sin
          }
          stage16_sw128(buf, lane, g * 16, lo);
          if (g < G1) {
            stage16_sw128(buf, lane, HALF + g * 16, hi);
          } else {
#pragma unroll
            for (int w = 0; w < 8; ++w) keep[g - G1][w] = hi[w];
          }
        }
        const CUtensorMap* map = kind == 0 ? tq : tk;
        store_box(map, 0, ty, h);
        if (DQK > 64) {
          buf = acquire();
#pragma unroll
          for (int g = G1; g < NG; ++g) stage16_sw128(buf, lane, HALF + g * 16 - 64, keep[g - G1]);
          store_box(map, 64, ty, h);
        }
      } else {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t raw[64];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld16(tacc + hh * 128 + hf * 64 + 16 * c, raw + 16 * c);
          tmem_ld_wait();
          if (last_head && hf == 1) release();
          const f2 sc = f2_make(sxw, sxw);
          uint8_t* buf = acquire();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = f2_to_bf16x2(
                  f2_mul(f2_make(__uint_as_float(raw[g * 16 + 2 * i]), __uint_as_float(raw[g * 16 + 2 * i + 1])), sc));
            stage16_sw128(buf, lane, g * 16, w);
          }
          store_box(tv, 64 * hf, ty, h);
        }
      }
    }
  }
};

// Epilogue warps and per-warp staging bytes of each GEMM.
constexpr int kFwdEW = 8, kDwEW = kDwEpiWarps;
constexpr int kFwdEPB = 4096, kDxEPB = 8192;

template <int DQK, bool PAIR>
__global__ void __launch_bounds__(gemm_threads(kFwdEW), 1)
    fwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBv,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ FwdParams p, DevStatus st,
                    Ring ring) {
  FwdSched sc{p, &tmBv, PAIR ? static_cast<int>(cluster_rank()) : 0, PAIR ? 2 : 1};
  FwdEpi<DQK> epi{p, sc, &tq, &tk, &tv, st};
  gemm_body<kFwdEW, kFwdEPB, PAIR>(sc, epi, &tmA, &tmB, ring, st, KID_FWD_GEMM);
}

// ---------------------------------------------------------------------------
// dX: schedule and epilogue
// ---------------------------------------------------------------------------
struct DxSched {
  static constexpr bool kMN = false;
  const DxParams& p;
  int rank, pair;
  __device__ int mtile(int u) const { return (u / p.n_tiles) * pair + rank; }
  // A: 128 tokens of dY8; B: one box of bn / pair rows of W8T (this CTA's
  // half of the tile's columns in a pair)
  template <bool PAIR>
  __device__ void load(const Unit& ui, int kb, const CUtensorMap* a, const CUtensorMap* b, uint8_t* sA,
                       uint8_t* sB, uint32_t bar) const {
    tma_load_2d_at<PAIR>(sA, a, bar, kb * kBK, ui.a_row);
    tma_load_2d_at<PAIR>(sB, b, bar, kb * kBK, ui.b_row);
  }
  __device__ int num_units() const { return p.num_units; }
  __device__ Unit unit(int u) const {
    Unit r;
    r.a_row = mtile(u) * kBM;
    r.b_row = (u % p.n_tiles) * p.bn + rank * (p.bn / pair);
    r.ncols = p.bn;
    r.b_bytes = p.bn / pair * kBK;
    r.b_sel = 0;
    r.kb0 = 0;
    r.kb1 = p.kblocks;
    return r;
  }
};

template <int MODE>
struct DxEpi {
  const DxParams& p;
  const DxSched& sc;
  const CUtensorMap* tdx;
  uint8_t* stage;
  int qw, sub, nsub, lane, ring;
  float scl;   // s_dy * s_w
  float k2;    // DRELU2: 2 sqrt(scale of the stored codes)
  float mx;    // RELU2 / DRELU2: running max |output| of this thread
  const float* sqrt_tab;   // DRELU2: sqrt of the E4M3 value of each code 0 .. 127
  // DRELU2: this thread's row of stored codes for the unit's columns (up to
  // 256), loaded by prepare() while the accumulator is still being computed
  static constexpr int kMaxChunks = 8;
  uint4 hc[kMaxChunks][2];
  __device__ void begin(int qw_, int sub_, int nsub_, int lane_, uint8_t* stage_) {
    qw = qw_;
    sub = sub_;
    nsub = nsub_;
    lane = lane_;
    stage = stage_;
    ring = 0;
    scl = (*p.dy_scale) * (*p.w_scale);
    mx = 0.f;
    if (MODE == EPI_DRELU2) {
      // sqrt(h^) = sqrt(code value) * sqrt(s_h): the stored squared activation
      // is non-negative, so its codes are 0 .. 0x7E and 128 square roots serve
      __shared__ float tab[128];
      const int i = (qw + 4 * sub) * 32 + lane;   // the epilogue warps fill the table
      if (i < 128) {
        float v = 0.f;
        if (i < 0x7F) {
          const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(i), __NV_E4M3);
          v = sqrtf(__half2float(*reinterpret_cast<const __half*>(&hr.x)));
        }
        tab[i] = v;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(dx_epi_warps(MODE) * 32) : "memory");
      sqrt_tab = tab;
      k2 = 2.f * sqrtf(*p.aux_scale);
    }
  }
  __device__ void finish() {
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
    if (MODE != EPI_PLAIN) {
      // rounding is monotone, so the bf16 of the max is the max of the bf16 outputs
      const float m = __bfloat162float(__float2bfloat16_rn(warp_max(mx)));
      if (lane == 0) p.amax_parts[blockIdx.x * dx_epi_warps(MODE) + qw + 4 * sub] = m;
    }
  }
  __device__ void prepare(int u) {
    if (MODE != EPI_DRELU2) return;
    const int t = sc.mtile(u) * kBM + qw * 32 + lane, j = u % p.n_tiles;
    const int share = p.bn / nsub;
    const uint4* src = reinterpret_cast<const uint4*>(p.aux8 + static_cast<int64_t>(t) * p.D + j * p.bn + sub * share);
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      hc[c][0] = hc[c][1] = make_uint4(0, 0, 0, 0);
      if (t < p.T && 32 * c < share) {
        hc[c][0] = __ldg(src + 2 * c);
        hc[c][1] = __ldg(src + 2 * c + 1);
      }
    }
  }
  __device__ void post(int) {}
  template <class Release>
  __device__ void process(int u, uint32_t tacc, Release& release) {
    const int m = sc.mtile(u), j = u % p.n_tiles;
    const int ty = m * kBM + qw * 32;
    const int share = p.bn / nsub;   // this warp's columns: [sub * share, (sub + 1) * share)
#pragma unroll
    for (int c = 0; c < kMaxChunks; ++c) {
      if (32 * c >= share) break;
      const int c0 = sub * share + 32 * c;
      uint8_t* slot = stage + (ring & 3) * 2048;
      if (lane == 0) bulk_wait_read<3>();
      __syncwarp();
      uint32_t raw[32];
      tmem_ld16(tacc + c0, raw);
      tmem_ld16(tacc + c0 + 16, raw + 16);
      tmem_ld_wait();
      if (32 * (c + 1) >= share) release();   // the last chunk's accumulator is read
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]) * scl;
      if (MODE == EPI_RELU2) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float r = fmaxf(v[i], 0.f);
          v[i] = r * r;
          mx = fmaxf(mx, v[i]);
        }
      } else if (MODE == EPI_DRELU2) {
        const uint32_t cw[8] = {hc[c][0].x, hc[c][0].y, hc[c][0].z, hc[c][0].w,
                                hc[c][1].x, hc[c][1].y, hc[c][1].z, hc[c][1].w};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = (v[i] * k2) * sqrt_tab[(cw[i >> 2] >> (8 * (i & 3))) & 0x7Fu];
          mx = fmaxf(mx, fabsf(v[i]));
        }
      }
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[g * 16 + 2 * i], v[g * 16 + 2 * i + 1]);
        stage16(slot, lane, g * 16, w);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0 && ty < p.T) {   // (a pair's second tile may lie wholly past T)
        tma_store_2d(tdx, slot, j * p.bn + c0, ty);
        bulk_commit();
      }
      ++ring;
    }
  }
};

template <bool PAIR, int MODE>
__global__ void __launch_bounds__(gemm_threads(dx_epi_warps(MODE)), 1)
    dx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tdx, const __grid_constant__ DxParams p, DevStatus st,
                   Ring ring) {
  DxSched sc{p, PAIR ? static_cast<int>(cluster_rank()) : 0, PAIR ? 2 : 1};
  DxEpi<MODE> epi{p, sc, &tdx};
  gemm_body<dx_epi_warps(MODE), kDxEPB, PAIR>(sc, epi, &tmA, &tmB, ring, st, KID_DX_GEMM);
}

// ---------------------------------------------------------------------------
// dW: split-K schedule, fp32 partial epilogue; the partials are summed in
// split order by dw_reduce_kernel, launched right after.
// dW = dY8^T . x8 reads both operands MN-major straight from the token-major
// tensors: a 128-token slice of dY8 [T, N] is the A tile (M = packed rows,
// contiguous) and of x8 [T, D] the B tile (N = model columns, contiguous).
// Token rows past T are zero-filled by TMA.
// ---------------------------------------------------------------------------
struct DwSched {
  static constexpr bool kMN = true;
  const DwParams& p;
  int rank, pair;
  // units: split-major over (pairs of) 128-row tiles of dW and bn-column tiles
  __device__ int tiles_per_split() const { return (p.m_tiles + pair - 1) / pair * p.n_tiles; }
  __device__ int split_of(int u) const { return u / tiles_per_split(); }
  __device__ int mtile(int u) const { return (u % tiles_per_split()) / p.n_tiles * pair + rank; }
  __device__ int ntile(int u) const { return (u % tiles_per_split()) % p.n_tiles; }
  // A: one box of 128 tokens x 128 packed columns at (a_row, k); B: this
  // CTA's bn / pair model columns as boxes of 128 tokens x 128 columns.
  template <bool PAIR>
  __device__ void load(const Unit& ui, int kb, const CUtensorMap* a, const CUtensorMap* b, uint8_t* sA,
                       uint8_t* sB, uint32_t bar) const {
    tma_load_2d_at<PAIR>(sA, a, bar, ui.a_row, kb * kBK);
    for (int j = 0; j < ui.ncols / pair / 128; ++j)
      tma_load_2d_at<PAIR>(sB + j * 16384, b, bar, ui.b_row + 128 * j, kb * kBK);
  }
  __device__ int num_units() const { return p.num_units; }
  __device__ Unit unit(int u) const {
    const int split = split_of(u);
    Unit r;
    r.a_row = mtile(u) * kBM;
    r.b_row = ntile(u) * p.bn + rank * (p.bn / pair);
    r.ncols = p.bn;
    r.b_bytes = p.bn / pair * kBK;
    r.b_sel = 0;
    r.kb0 = static_cast<int>(static_cast<int64_t>(split) * p.kblocks_total / p.splits);
    r.kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * p.kblocks_total / p.splits);
    return r;
  }
};

// Epilogue of the dW GEMM.  Each unit stores its fp32 partial tile in the
// layout [bn / 4][128 rows][4 columns], so that both the stores here and the
// loads of the reduction kernel are 16 bytes per lane and coalesced; an
// epilogue warp stores one sub-tile (32 rows x bn / nsub columns).  (Summing
// the splits here, in whichever warp stored a sub-tile's last split, left a
// 10 us tail of dependent loads at the end of the kernel; a kernel of its own
// spreads the sum over the whole GPU.)
struct DwEpi {
  const DwParams& p;
  const DwSched& sc;
  int qw, sub, nsub, lane;
  __device__ void begin(int qw_, int sub_, int nsub_, int lane_, uint8_t*) {
    qw = qw_;
    sub = sub_;
    nsub = nsub_;
    lane = lane_;
  }
  __device__ void finish() {}
  __device__ void prepare(int) {}
  __device__ int64_t tile_of(int u, int split) const {
    return (static_cast<int64_t>(split) * p.m_tiles + sc.mtile(u)) * p.n_tiles + sc.ntile(u);
  }
  // float4 index of columns [c, c + 4) of row `row` inside a partial tile
  __device__ static int quad(int c, int row) { return (c >> 2) * kBM + row; }
  template <class Release>
  __device__ void process(int u, uint32_t tacc, Release& release) {
    // the odd CTA of the last pair may lie past the rows
    if (sc.mtile(u) >= p.m_tiles) return;
    const int row = qw * 32 + lane;
    float4* dst = reinterpret_cast<float4*>(p.partials + tile_of(u, sc.split_of(u)) * p.bn * kBM);
    const int share = p.bn / nsub;
    for (int c0 = sub * share; c0 < (sub + 1) * share; c0 += 32) {
      uint32_t raw[32];
      tmem_ld16(tacc + c0, raw);
      tmem_ld16(tacc + c0 + 16, raw + 16);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[quad(c0 + 4 * i, row)] = make_float4(__uint_as_float(raw[4 * i]), __uint_as_float(raw[4 * i + 1]),
                                                 __uint_as_float(raw[4 * i + 2]), __uint_as_float(raw[4 * i + 3]));
    }
    release();   // the accumulator is read
  }
  __device__ void post(int) {}
};

template <bool PAIR>
__global__ void __launch_bounds__(gemm_threads(kDwEW), 1)
    dw_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ DwParams p, DevStatus st, Ring ring) {
  DwSched sc{p, PAIR ? static_cast<int>(cluster_rank()) : 0, PAIR ? 2 : 1};
  DwEpi epi{p, sc};
  gemm_body<kDwEW, 0, PAIR>(sc, epi, &tmA, &tmB, ring, st, KID_DW_GEMM);
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
// Every GEMM kernel may use up to kSmemMax bytes of dynamic shared memory.
template <class K>
static cudaError_t set_smem_once(K kernel, std::atomic<bool> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
  if (e == cudaSuccess && dev < 64) done[dev].store(true, std::memory_order_relaxed);
  return e;
}

// Co-resident 2-CTA clusters of a kernel at a given shared-memory size,
// queried once per (kernel, device, size): per device one word holding the
// size (high half) and the count (low half), so that a reader never pairs
// one call's size with another's count.
struct ClusterCache {
  std::atomic<uint64_t> v[64];
  int lookup(int dev, int smem) const {
    if (dev >= 64) return 0;
    const uint64_t w = v[dev].load(std::memory_order_relaxed);
    return static_cast<int>(w >> 32) == smem ? static_cast<int>(w & 0xFFFFFFFFu) : 0;
  }
  void store(int dev, int smem, int clusters) {
    if (dev < 64)
      v[dev].store((static_cast<uint64_t>(static_cast<uint32_t>(smem)) << 32) | static_cast<uint32_t>(clusters),
                   std::memory_order_relaxed);
  }
};

// Persistent launch: one CTA per SM (at most one per unit), or for pairs one
// 2-CTA cluster per co-resident pair of SMs (at most one per unit).
template <class... KArgs, class... Args>
static cudaError_t launch_persistent(void (*kernel)(KArgs...), bool pair, int units, int sms, int threads, int smem,
                                     ClusterCache& cache, int* grid_used, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  int grid = units < sms ? units : sms;
  if (pair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int clusters = cache.lookup(dev, smem);
    if (clusters <= 0) {
      cfg.gridDim = dim3(2 * (sms / 2 > 0 ? sms / 2 : 1));
      e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters <= 0) return cudaErrorInvalidConfiguration;
      cache.store(dev, smem, clusters);
    }
    grid = 2 * (units < clusters ? units : clusters);
  }
  cfg.gridDim = dim3(grid);
  if (grid_used) *grid_used = grid;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int DQK, bool PAIR>
static cudaError_t launch_fwd_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBv,
                                const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                                int sms, DevStatus st, cudaStream_t s) {
  static std::atomic<bool> done[64];
  static ClusterCache cache;
  // B tiles: hq heads of q or k, or two heads of v (this CTA's half in a pair)
  const int brows = (p.hq * DQK > 2 * p.d_v ? p.hq * DQK : 2 * p.d_v) / p.pair;
  const Ring ring = ring_for(brows * kBK, kFwdEW, kFwdEPB);
  cudaError_t e = set_smem_once(fwd_gemm_kernel<DQK, PAIR>, done);
  if (e != cudaSuccess) return e;
  return launch_persistent(fwd_gemm_kernel<DQK, PAIR>, PAIR, p.num_units, sms, gemm_threads(kFwdEW),
                           gemm_smem_bytes(ring, kFwdEW, kFwdEPB), cache, nullptr, s, tmA, tmB, tmBv, tq, tk, tv, p, st,
                           ring);
}

template <bool PAIR>
static cudaError_t launch_fwd_p(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBv,
                                const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                                int sms, DevStatus st, cudaStream_t s) {
  switch (p.d_qk) {
    case 64: return launch_fwd_t<64, PAIR>(tmA, tmB, tmBv, tq, tk, tv, p, sms, st, s);
    case 96: return launch_fwd_t<96, PAIR>(tmA, tmB, tmBv, tq, tk, tv, p, sms, st, s);
    case 128: return launch_fwd_t<128, PAIR>(tmA, tmB, tmBv, tq, tk, tv, p, sms, st, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBv,
                            const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                            int sms, DevStatus st, cudaStream_t s) {
  return p.pair == 2 ? launch_fwd_p<true>(tmA, tmB, tmBv, tq, tk, tv, p, sms, st, s)
                     : launch_fwd_p<false>(tmA, tmB, tmBv, tq, tk, tv, p, sms, st, s);
}

template <bool PAIR, int MODE>
static cudaError_t launch_dx_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tdx,
                               const DxParams& p, int sms, DevStatus st, cudaStream_t s, int* grid_used) {
  static std::atomic<bool> done[64];
  static ClusterCache cache;
  constexpr int EW = dx_epi_warps(MODE);
  const Ring ring = ring_for(p.bn / p.pair * kBK, EW, kDxEPB);
  cudaError_t e = set_smem_once(dx_gemm_kernel<PAIR, MODE>, done);
  if (e != cudaSuccess) return e;
  return launch_persistent(dx_gemm_kernel<PAIR, MODE>, PAIR, p.num_units, sms, gemm_threads(EW),
                           gemm_smem_bytes(ring, EW, kDxEPB), cache, grid_used, s, tmA, tmB, tdx, p, st, ring);
}

template <bool PAIR>
static cudaError_t launch_dx_m(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tdx,
                               const DxParams& p, int sms, DevStatus st, cudaStream_t s, int* grid_used) {
  switch (p.mode) {
    case EPI_PLAIN: return launch_dx_t<PAIR, EPI_PLAIN>(tmA, tmB, tdx, p, sms, st, s, grid_used);
    case EPI_RELU2: return launch_dx_t<PAIR, EPI_RELU2>(tmA, tmB, tdx, p, sms, st, s, grid_used);
    case EPI_DRELU2: return launch_dx_t<PAIR, EPI_DRELU2>(tmA, tmB, tdx, p, sms, st, s, grid_used);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dx_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tdx,
                           const DxParams& p, int sms, DevStatus st, cudaStream_t s, int* grid_used) {
  return p.pair == 2 ? launch_dx_m<true>(tmA, tmB, tdx, p, sms, st, s, grid_used)
                     : launch_dx_m<false>(tmA, tmB, tdx, p, sms, st, s, grid_used);
}

template <bool PAIR>
static cudaError_t launch_dw_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const DwParams& p, int sms,
                               DevStatus st, cudaStream_t s) {
  static std::atomic<bool> done[64];
  static ClusterCache cache;
  const Ring ring = ring_for(p.bn / p.pair * kBK, kDwEW, 0);
  cudaError_t e = set_smem_once(dw_gemm_kernel<PAIR>, done);
  if (e != cudaSuccess) return e;
  return launch_persistent(dw_gemm_kernel<PAIR>, PAIR, p.num_units, sms, gemm_threads(kDwEW),
                           gemm_smem_bytes(ring, kDwEW, 0), cache, nullptr, s, tmA, tmB, p, st, ring);
}

// Sum of the dW GEMM's split partials, in split order (the same sum on every
// run), scaled by s_dy * s_x and stored as bf16.  A warp takes 8 rows x 8
// column quads, a lane two quads of one row (all their splits' loads in
// flight together): each load instruction reads four 128-byte runs (8
// consecutive rows of one quad), each store 32 bytes of a row.
__global__ void __launch_bounds__(256) dw_reduce_kernel(const __grid_constant__ DwParams p) {
  constexpr int kMaxS = 4;   // splits whose loads are issued together
  const int lane = threadIdx.x & 31;
  const int qblocks = p.D / 32;                                   // 8-quad blocks along D
  const int64_t tiles = static_cast<int64_t>((p.N + 7) / 8) * qblocks;
  const float scl = (*p.dy_scale) * (*p.x_scale);
  const int64_t split_stride = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.bn * kBM / 4;   // float4s
  const float4* src = reinterpret_cast<const float4*>(p.partials);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < tiles; w += nwarps) {
    const int n = static_cast<int>(w / qblocks) * 8 + (lane & 7);
    if (n >= p.N) continue;
    const int mt = n / kBM, row = n % kBM;
    int64_t at[2];
    int d[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      d[h] = (static_cast<int>(w % qblocks) * 8 + (lane >> 3) + 4 * h) * 4;
      const int nt = d[h] / p.bn, c = d[h] % p.bn;
      at[h] = (static_cast<int64_t>(mt) * p.n_tiles + nt) * p.bn * kBM / 4 + (c / 4) * kBM + row;
    }
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int s0 = 0; s0 < p.splits; s0 += kMaxS) {
      float4 v[kMaxS][2];
#pragma unroll
      for (int j = 0; j < kMaxS; ++j)
        if (s0 + j < p.splits)
#pragma unroll
          for (int h = 0; h < 2; ++h) v[j][h] = __ldcg(src + (s0 + j) * split_stride + at[h]);
#pragma unroll
      for (int j = 0; j < kMaxS; ++j)
        if (s0 + j < p.splits)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            acc[h].x += v[j][h].x;
            acc[h].y += v[j][h].y;
            acc[h].z += v[j][h].z;
            acc[h].w += v[j][h].w;
          }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<uint2*>(p.dW + static_cast<int64_t>(n) * p.D + d[h]) =
          make_uint2(pack_bf16x2(acc[h].x * scl, acc[h].y * scl), pack_bf16x2(acc[h].z * scl, acc[h].w * scl));
  }
}

cudaError_t launch_dw_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const DwParams& p, int sms,
                           DevStatus st, cudaStream_t s) {
  cudaError_t e =
      p.pair == 2 ? launch_dw_t<true>(tmA, tmB, p, sms, st, s) : launch_dw_t<false>(tmA, tmB, p, sms, st, s);
  if (e != cudaSuccess) return e;
  const int64_t tiles = static_cast<int64_t>((p.N + 7) / 8) * (p.D / 32);
  const int64_t blocks = (tiles + 7) / 8;   // eight warps per block
  const int grid = static_cast<int>(blocks < 8 * sms ? blocks : 8 * sms);
  dw_reduce_kernel<<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace qkvp

// Argument blocks and host-side launchers of the qkvp kernels.  Every
// launcher enqueues on `stream` and returns the cudaError_t of the launch.
#pragma once

#include "common.cuh"

namespace qkvp {

constexpr int kMaxLayers = 128;

// Host-side helpers of the C ABI shared by its translation units.
// check_dims: QKVP_OK or the status the entry points return for `d`.
int check_dims(const qkvp_dims* d);
// mark: records the next armed timing event (qkvp_set_timing_events) on `s`.
void mark(cudaStream_t s);

// ---------------------------------------------------------------------------
// Bank refresh
// ---------------------------------------------------------------------------
struct BankArgs {
  const uint16_t* Wq[kMaxLayers];
  const uint16_t* Wk[kMaxLayers];
  const uint16_t* Wv[kMaxLayers];
  uint8_t* W8;       // [L, N, D]
  uint8_t* W8T;      // [L, D, N]
  float* w_scale;    // [L]
  int L, D, N, Nq;   // Nq = H * d_qk
};
// Counters of one bank refresh, in device memory that starts at zero; the
// refresh kernel leaves them at zero when it completes.
struct BankSync {
  unsigned int next;               // work items claimed
  unsigned int exited;             // blocks past their last item
  unsigned int amax[kMaxLayers];   // per layer: bit pattern of max |w| so far
  unsigned int done[kMaxLayers];   // per layer: amax items finished
  unsigned int scale[kMaxLayers];  // per layer: bit pattern of the scale once known, else 0
};

// Amax and both code layouts of every layer in one launch (any grid size
// works: blocks claim work items from the counters in `sy`).
cudaError_t launch_bank_refresh(const BankArgs& a, BankSync* sy, DevStatus st, cudaStream_t s);

// ---------------------------------------------------------------------------
// Activation quantisation
// ---------------------------------------------------------------------------
// amax of n bf16 values at x (16-byte aligned); writes `blocks` partials.
cudaError_t launch_amax_bf16(const uint16_t* x, int64_t n, float* partials, int blocks, cudaStream_t s);
// x (n bf16, n % 16 == 0) -> x8 codes and x_scale; reads `nparts` partials.
cudaError_t launch_x_quant(const uint16_t* x, int64_t n, uint8_t* x8, const float* partials, int nparts,
                           float* x_scale, int blocks, cudaStream_t s);

// A grid-wide barrier between the blocks of one launch, in device memory
// that starts at zero and is left at zero-count after every use.
struct GridBar {
  int count;   // blocks arrived in the current use
  int gen;     // uses completed (the waiters watch it change)
};
// Both steps in one persistent launch: amax of x (one partial per block, at
// most kMaxFusedBlocks), a grid barrier, then every block reduces the
// partials and quantises the same elements it read (mostly from L2 when x
// fits there).  Every block must be resident at once: the grid is sized from
// the occupancy of the kernel; the barrier's wait is bounded.
constexpr int kMaxFusedBlocks = 4096;
cudaError_t launch_x_amax_quant(const uint16_t* x, int64_t n, uint8_t* x8, float* partials, float* x_scale,
                                GridBar* bar, DevStatus st, cudaStream_t s);

cudaError_t launch_rope_table(float* table, int max_pos, int d_qk, double base, cudaStream_t s);
cudaError_t launch_selftest_wait(DevStatus st, cudaStream_t s);

// ---------------------------------------------------------------------------
// GEMMs (tcgen05, E4M3 operands via TMA).  With pair = 2 a unit is a 256-row
// tile computed by a 2-CTA cluster (one MMA per K step over both CTAs'
// shared memory); with pair = 1 a 128-row tile computed by one CTA.
// ---------------------------------------------------------------------------
constexpr int kMaxFwdTiles = 192;   // 2 * 64 q/k tiles + 64 v tiles at H = 128
struct FwdParams {
  int T, H, d_qk, d_v;
  int hq;            // heads per Q (or K) tile
  int nq;            // Q tiles (= K tiles) per 128-token block
  int nv;            // V tiles per block (2 heads each)
  int n_tiles;       // 2*nq + nv
  // tile of each slot of a token block: q, v and k tiles interleaved in
  // proportion, so that a CTA's consecutive units alternate between the
  // q/k epilogue (norm and rotation) and the lighter v one
  uint8_t tile_order[kMaxFwdTiles];
  int pair;          // CTAs per unit (1 or 2)
  int num_units;     // ceil(ceil(T/128) / pair) * n_tiles
  int kblocks;       // D / 128
  float eps;
  const float* x_scale;
  const float* w_scale;
  const float* rope;  // [d_qk/4][max_pos] (cos, cos, sin, sin) of two rotation pairs
  int max_pos;
  const int32_t* pos;
  float* rstd;        // [2, H, T]
};

// Epilogues of the dX-shaped GEMM (out = A . B^T * sa * sb, bf16):
//   EPI_PLAIN   the scaled product
//   EPI_RELU2   relu(v)^2 of the scaled product v, plus per-warp amax partials
//   EPI_DRELU2  v * 2 sqrt(h^) with h^ the de-quantised codes aux8 (same
//               [T, D] layout as the output) times aux_scale, plus per-warp
//               amax partials (the ReLU-squared backward, relu(pre) rebuilt
//               from the stored squared activation)
enum EpiMode : int { EPI_PLAIN = 0, EPI_RELU2 = 1, EPI_DRELU2 = 2 };

struct DxParams {
  int T, D, bn, n_tiles, pair, num_units, kblocks;   // num_units = ceil(ceil(T/128) / pair) * n_tiles
  const float* dy_scale;
  const float* w_scale;
  int mode;                // EpiMode
  float* amax_parts;       // RELU2 / DRELU2: [grid * dx_epi_warps(mode)] max |output| (bf16-rounded) per CTA and epilogue warp
  const uint8_t* aux8;     // DRELU2: [T, D] E4M3 codes
  const float* aux_scale;  // DRELU2: their scale
};

// Epilogue warps of the dW GEMM.
constexpr int kDwEpiWarps = 8;
// Epilogue warps of the dX-shaped GEMM per epilogue mode (the ReLU-squared
// modes do more per element and take eight); each writes one amax partial in
// the RELU2 / DRELU2 modes.
__host__ __device__ constexpr int dx_epi_warps(int mode) { return mode == EPI_PLAIN ? 4 : 8; }

struct DwParams {
  // num_units = splits * ceil(m_tiles / pair) * n_tiles; kblocks_total = ceil(T/128)
  int N, D, bn, m_tiles, n_tiles, pair, splits, num_units, kblocks_total;
  float* partials;    // [splits][m_tiles][n_tiles] tiles of [bn / 4][128][4] float32
  const float* dy_scale;
  const float* x_scale;
  uint16_t* dW;       // [N, D] bf16
};

// Persistent launches sized to the device (`sms` multiprocessors).
// tmB / tmBv: W8 with box heights hq*d_qk/pair (q/k tiles) and 2*d_v/pair (v
// tiles); dX: W8T with box height bn/pair.
cudaError_t launch_fwd_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBv,
                            const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                            int sms, DevStatus st, cudaStream_t s);
// *grid_used (if non-null) receives the launch's grid (amax partials:
// dx_epi_warps(mode) per CTA).
cudaError_t launch_dx_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tdx,
                           const DxParams& p, int sms, DevStatus st, cudaStream_t s, int* grid_used = nullptr);
cudaError_t launch_dw_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const DwParams& p, int sms,
                           DevStatus st, cudaStream_t s);


// ---------------------------------------------------------------------------
// Backward epilogue (norm/RoPE backward, dY amax, dY quantisation)
// ---------------------------------------------------------------------------
struct BwdParams {
  int T, H, d_qk, d_v, N, tiles, num_units;
  const float* rstd;     // [2, H, T]
  const int32_t* pos;
  const float* rope;
  int max_pos;
  float* partials;       // amax partials (written by pass 1, read by pass 2)
  int nparts;            // grid of pass 1
  float* dy_scale;       // written by pass 2
  float* mu;             // [2, H, T] mean(g_out * o) of every q/k row: pass 1 writes it, pass 2 reads it
};
// Tokens per work unit of the backward epilogue (the height of its TMA boxes).
constexpr int kBwdUnitRows = 64;
struct BwdMaps {
  CUtensorMap dq, q, dk, k, dv;   // loads, 3-D [H][T][d], box {32, kBwdUnitRows, 1}, 64-byte swizzle
  CUtensorMap dy8;                // store: [T][N] codes, box {32, kBwdUnitRows}, 32-byte swizzle
};
cudaError_t launch_bwd_amax(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s);
cudaError_t launch_bwd_quant(const BwdMaps& m, const BwdParams& p, int grid, DevStatus st, cudaStream_t s);

}  // namespace qkvp

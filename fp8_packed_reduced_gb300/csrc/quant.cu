// Bandwidth-bound quantisation kernels:
//   bank refresh  (amax per layer, then codes in both layouts from one pass)
//   x amax        (per-tensor amax of the activations)
//   x quantise    (codes of x, token-major)
//   RoPE table, and the timeout self-test kernel.
#include <algorithm>
#include <atomic>

#include "kernels.cuh"

namespace qkvp {

// ---------------------------------------------------------------------------
// Per-tensor amax of a bf16 tensor: one partial maximum per block.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float absmax_bf16x8(uint4 w) {
  float m = 0.f;
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(bf16_lo(u[i])));
    m = fmaxf(m, fabsf(bf16_hi(u[i])));
  }
  return m;
}

// x: n16 groups of 8 bf16 (16 bytes) followed by `tail` (< 8) bf16 values.
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint16_t* __restrict__ x, int64_t n16, int tail,
                                                         float* __restrict__ partials) {
  __shared__ float red[32];
  const uint4* p = reinterpret_cast<const uint4*>(x);
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < n16; i += 8 * stride) {  // eight independent loads in flight
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldg(p + i + j * stride);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, absmax_bf16x8(v[j]));
  }
  for (; i < n16; i += stride) m = fmaxf(m, absmax_bf16x8(__ldg(p + i)));
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail)
    m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[n16 * 8 + threadIdx.x]) << 16)));
  m = block_max(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

cudaError_t launch_amax_bf16(const uint16_t* x, int64_t n, float* partials, int blocks, cudaStream_t s) {
  amax_bf16_kernel<<<blocks, 256, 0, s>>>(x, n / 8, static_cast<int>(n % 8), partials);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bank refresh.  Pass 1: amax of each layer's logical Q/K/V packs, read in
// place (no concatenation).  Pass 2: every block re-reduces its layer's
// partials, then converts 128 x 128 tiles of the bank and writes each to both
// W8 (row-major) and W8T (transposed) from the one read of that tile.  All
// layers of a refresh go in one launch per pass, each sized to one wave; the
// second pass reads the bank back from L2 for bank sizes that fit there.
// ---------------------------------------------------------------------------
__device__ __forceinline__ const uint16_t* bank_row(const BankArgs& a, int l, int n) {
  if (n < a.Nq) return a.Wq[l] + static_cast<int64_t>(n) * a.D;
  if (n < 2 * a.Nq) return a.Wk[l] + static_cast<int64_t>(n - a.Nq) * a.D;
  return a.Wv[l] + static_cast<int64_t>(n - 2 * a.Nq) * a.D;
}

// grid: (kBankAmaxBlocks, L), 1024 threads.  Block b of layer l takes a
// contiguous band of rows; one warp per row, two rows in flight, the lanes
// over the row's 16-byte chunks.
__global__ void __launch_bounds__(1024) bank_amax_kernel(const __grid_constant__ BankArgs a, float* partials) {
  __shared__ float red[32];
  const int l = blockIdx.y;
  const int cpr = a.D / 8;   // 16-byte chunks per row
  const int band = (a.N + gridDim.x - 1) / gridDim.x;
  const int r0 = blockIdx.x * band, r1 = min(a.N, r0 + band);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float m = 0.f;
  int n = r0 + warp;
  for (; n + nw < r1; n += 2 * nw) {
    const uint4* ra = reinterpret_cast<const uint4*>(bank_row(a, l, n));
    const uint4* rb = reinterpret_cast<const uint4*>(bank_row(a, l, n + nw));
#pragma unroll 4
    for (int c = lane; c < cpr; c += 32)
      m = fmaxf(m, fmaxf(absmax_bf16x8(__ldg(ra + c)), absmax_bf16x8(__ldg(rb + c))));
  }
  if (n < r1) {
    const uint4* ra = reinterpret_cast<const uint4*>(bank_row(a, l, n));
#pragma unroll 4
    for (int c = lane; c < cpr; c += 32) m = fmaxf(m, absmax_bf16x8(__ldg(ra + c)));
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) partials[l * gridDim.x + blockIdx.x] = m;
}

// Transpose of a 4 x 4 byte block held as four row words: out[c] = bytes
// (r0[c], r1[c], r2[c], r3[c]).
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t (&out)[4]) {
  const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);   // (r0c0 r1c0 r0c1 r1c1), (.. c2 .. c3)
  const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

// grid: (ceil(N/128) * D/128, L); 256 threads; tile 128 rows x 128 columns.
// Thread t converts rows 4 (t / 8) .. + 3, columns 16 (t % 8) .. + 15 of the
// tile: one 16-byte code store per row into W8, and, transposed in registers
// by 4 x 4 byte blocks, sixteen 4-byte column words into a shared tile [128
// columns][32 words of 4 rows], whose word index is XORed with 4 * (column /
// 16) % 32 so that a warp's stores hit 32 banks; the tile then leaves as
// 16-byte chunks of W8T rows.
__global__ void __launch_bounds__(256) bank_quant_kernel(const __grid_constant__ BankArgs a,
                                                         const float* partials) {
  __shared__ float red[32];
  __shared__ __align__(16) uint32_t tr[128][32];   // [tile column][row group, swizzled]
  const int l = blockIdx.y;
  const int tiles_d = a.D / 128;
  const int tiles = (a.N + 127) / 128 * tiles_d;
  const float amax = block_reduce_partials(partials + l * kBankAmaxBlocks, kBankAmaxBlocks, red);
  const float s = scale_from_amax(amax);
  const Bracket2 k = make_bracket2(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) a.w_scale[l] = s;

  const int rg = threadIdx.x >> 3, cg = threadIdx.x & 7;
  uint8_t* W8 = a.W8 + static_cast<int64_t>(l) * a.N * a.D;
  uint8_t* W8T = a.W8T + static_cast<int64_t>(l) * a.N * a.D;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {   // the layer's tiles, round-robin
  const int n0 = (tile / tiles_d) * 128, d0 = (tile % tiles_d) * 128;
  if (tile != static_cast<int>(blockIdx.x)) __syncthreads();   // the previous tile has left `tr`
  uint4 code[4];   // the four rows' 16 codes
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + 4 * rg + i;
    if (n < a.N) {
      const uint4* src = reinterpret_cast<const uint4*>(bank_row(a, l, n) + d0 + 16 * cg);
      const uint4 u0 = __ldg(src), u1 = __ldg(src + 1);
      const f2 v0[4] = {f2_from_bf16x2(u0.x), f2_from_bf16x2(u0.y), f2_from_bf16x2(u0.z), f2_from_bf16x2(u0.w)};
      const f2 v1[4] = {f2_from_bf16x2(u1.x), f2_from_bf16x2(u1.y), f2_from_bf16x2(u1.z), f2_from_bf16x2(u1.w)};
      const uint2 c0 = quant8(v0, k), c1 = quant8(v1, k);
      code[i] = make_uint4(c0.x, c0.y, c1.x, c1.y);
      *reinterpret_cast<uint4*>(W8 + static_cast<int64_t>(n) * a.D + d0 + 16 * cg) = code[i];
    } else {
      code[i] = make_uint4(0, 0, 0, 0);
    }
  }
  // column 16 cg + 4 q + c holds the bytes of rows 4 rg .. 4 rg + 3
  const int sw = (cg & 7) << 2;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[4];
    const uint32_t* r = reinterpret_cast<const uint32_t*>(code);
    transpose4x4(r[q], r[4 + q], r[8 + q], r[12 + q], w);
#pragma unroll
    for (int c = 0; c < 4; ++c) tr[16 * cg + 4 * q + c][rg ^ sw] = w[c];
  }
  __syncthreads();
  // W8T rows d0 .. d0 + 127, columns n0 .. n0 + 127 (N is a multiple of 64):
  // chunk i (rows 16 i .. 16 i + 15 of the tile) of column col is the word
  // group 4 i .. 4 i + 3, stored at 4 (i ^ (col / 16 % 8)).
  const int nvalid = min(128, a.N - n0);
  for (int e = threadIdx.x; e < 128 * 8; e += 256) {
    const int col = e >> 3, i = e & 7;
    if (16 * i < nvalid) {
      const uint4 val = *reinterpret_cast<const uint4*>(&tr[col][4 * (i ^ ((col >> 4) & 7))]);
      *reinterpret_cast<uint4*>(W8T + static_cast<int64_t>(d0 + col) * a.N + n0 + 16 * i) = val;
    }
  }
  }
}

static int bank_sms() {
  static std::atomic<int> cache[64];   // per device, written once
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

// Up to 9 layers the amax grid fits the GPU in one wave of 1024-thread
// blocks (two per SM); beyond that, blocks of 512 threads keep it to one.
cudaError_t launch_bank_amax(const BankArgs& a, float* partials, cudaStream_t s) {
  const int sms = bank_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int threads = kBankAmaxBlocks * a.L <= 2 * sms ? 1024 : 512;
  bank_amax_kernel<<<dim3(kBankAmaxBlocks, a.L), threads, 0, s>>>(a, partials);
  return cudaGetLastError();
}

// One block per tile while the tiles of all layers fit on the GPU at once;
// beyond that each block takes several tiles of its layer (one wave).
cudaError_t launch_bank_quant(const BankArgs& a, const float* partials, cudaStream_t s) {
  static std::atomic<int> per_sm[64];   // per device, written once
  const int sms = bank_sms();
  if (sms <= 0) return cudaErrorInvalidDevice;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int resident = dev < 64 ? per_sm[dev].load(std::memory_order_relaxed) : 0;
  if (resident <= 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, bank_quant_kernel, 256, 0);
    if (e != cudaSuccess) return e;
    if (resident < 1) return cudaErrorInvalidConfiguration;
    if (dev < 64) per_sm[dev].store(resident, std::memory_order_relaxed);
  }
  const int tiles = ((a.N + 127) / 128) * (a.D / 128);
  const int per_layer = std::max(1, std::min(tiles, resident * sms / a.L));
  bank_quant_kernel<<<dim3(per_layer, a.L), 256, 0, s>>>(a, partials);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// x -> x8 [T, D] codes.  Every block first re-reduces the amax partials of
// x (a few KB from L2), then converts 16 values per thread per step: two
// 16-byte loads, one 16-byte store.  T * D is a multiple of 16 (D % 128 == 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 quant16(uint4 u0, uint4 u1, const Bracket& k) {
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  uint32_t q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    q[j] = quant4_fast(bf16_lo(w[2 * j]), bf16_hi(w[2 * j]), bf16_lo(w[2 * j + 1]), bf16_hi(w[2 * j + 1]), k);
  return make_uint4(q[0], q[1], q[2], q[3]);
}

__global__ void __launch_bounds__(256) x_quant_kernel(const uint16_t* __restrict__ x, int64_t n16,
                                                      uint8_t* __restrict__ x8, const float* partials, int nparts,
                                                      float* x_scale) {
  __shared__ float red[32];
  const float s = scale_from_amax(block_reduce_partials(partials, nparts, red));
  const Bracket k = make_bracket(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *x_scale = s;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(x8);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + stride < n16; i += 2 * stride) {  // two independent groups in flight
    const uint4 a0 = __ldg(src + 2 * i), a1 = __ldg(src + 2 * i + 1);
    const uint4 b0 = __ldg(src + 2 * (i + stride)), b1 = __ldg(src + 2 * (i + stride) + 1);
    dst[i] = quant16(a0, a1, k);
    dst[i + stride] = quant16(b0, b1, k);
  }
  for (; i < n16; i += stride) dst[i] = quant16(__ldg(src + 2 * i), __ldg(src + 2 * i + 1), k);
}

cudaError_t launch_x_quant(const uint16_t* x, int64_t n, uint8_t* x8, const float* partials, int nparts,
                           float* x_scale, int blocks, cudaStream_t s) {
  x_quant_kernel<<<blocks, 256, 0, s>>>(x, n / 16, x8, partials, nparts, x_scale);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// x amax and x quantise in one launch, separated by a grid barrier.
// ---------------------------------------------------------------------------
// Grid barrier: every block's thread 0 arrives; the last to arrive resets the
// count and advances the generation, the others wait (bounded) for that.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void grid_barrier(GridBar* bar, const DevStatus& st, int kid) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const int gen = ld_acquire_gpu(&bar->gen);
    __threadfence();   // this block's writes before its arrival
    if (atomicAdd(&bar->count, 1) == static_cast<int>(gridDim.x) - 1) {
      bar->count = 0;
      __threadfence();
      atomicAdd(&bar->gen, 1);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(&bar->gen) == gen) {
        if (globaltimer_ns() - t0 > st.timeout_ns) {
          record_error(st, QKVP_ERR_TIMEOUT, kid);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

constexpr int kFusedThreads = 512;

// 16-byte read-only load with an L2 eviction-priority policy (createpolicy).
__device__ __forceinline__ uint4 ldg_hint(const uint4* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

__global__ void __launch_bounds__(kFusedThreads) x_amax_quant_kernel(const uint16_t* __restrict__ x, int64_t n16,
                                                                     uint8_t* __restrict__ x8, float* partials,
                                                                     float* x_scale, GridBar* bar, DevStatus st) {
  __shared__ float red[32];
  const uint4* src = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // 1: amax over this block's groups of 16 values (four groups in flight);
  // the lines are kept in L2 with priority for step 2
  const uint64_t keep = l2_policy_evict_last();
  float m = 0.f;
  int64_t i = i0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = ldg_hint(src + 2 * (i + j * stride), keep);
      v[2 * j + 1] = ldg_hint(src + 2 * (i + j * stride) + 1, keep);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, absmax_bf16x8(v[j]));
  }
  for (; i < n16; i += stride)
    m = fmaxf(m, fmaxf(absmax_bf16x8(ldg_hint(src + 2 * i, keep)), absmax_bf16x8(ldg_hint(src + 2 * i + 1, keep))));
  m = block_max(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
  grid_barrier(bar, st, KID_X_QUANT);
  // 2: the scale from every block's partial, then the codes of the same groups
  float pm = 0.f;   // the other blocks' partials, read from L2
  for (int b = threadIdx.x; b < static_cast<int>(gridDim.x); b += blockDim.x) pm = fmaxf(pm, __ldcg(partials + b));
  const float s = scale_from_amax(block_max(pm, red));
  const Bracket k = make_bracket(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *x_scale = s;
  // in the reverse order of step 1: the groups read last are the likeliest
  // to be in L2 still
  // (last use of the lines: they may go first)
  const uint64_t done = l2_policy_evict_first();
  uint4* dst = reinterpret_cast<uint4*>(x8);
  const int64_t cnt = i0 < n16 ? (n16 - 1 - i0) / stride + 1 : 0;   // this thread's groups
  int64_t c = cnt - 1;
  for (; c >= 1; c -= 2) {
    const int64_t ia = i0 + c * stride, ib = ia - stride;
    const uint4 a0 = ldg_hint(src + 2 * ia, done), a1 = ldg_hint(src + 2 * ia + 1, done);
    const uint4 b0 = ldg_hint(src + 2 * ib, done), b1 = ldg_hint(src + 2 * ib + 1, done);
    dst[ia] = quant16(a0, a1, k);
    dst[ib] = quant16(b0, b1, k);
  }
  if (c == 0) dst[i0] = quant16(ldg_hint(src + 2 * i0, done), ldg_hint(src + 2 * i0 + 1, done), k);
}

cudaError_t launch_x_amax_quant(const uint16_t* x, int64_t n, uint8_t* x8, float* partials, float* x_scale,
                                GridBar* bar, DevStatus st, cudaStream_t s) {
  static std::atomic<int> cache[64];   // per device, written once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int blocks = dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (blocks <= 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, x_amax_quant_kernel, kFusedThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    blocks = sms * per_sm < kMaxFusedBlocks ? sms * per_sm : kMaxFusedBlocks;
    if (dev < 64) cache[dev].store(blocks, std::memory_order_relaxed);
  }
  // no more blocks than groups of 16 values (each block then has work in both steps)
  const int64_t n16 = n / 16;
  const int grid = static_cast<int>(n16 < blocks ? (n16 > 0 ? n16 : 1) : blocks);
  x_amax_quant_kernel<<<grid, kFusedThreads, 0, s>>>(x, n16, x8, partials, x_scale, bar, st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RoPE table, two rotation pairs per entry:
//   table[(j * max_pos + p) * 4 + {0, 1, 2, 3}]
//     = cos(p w_2j), cos(p w_2j+1), sin(p w_2j), sin(p w_2j+1),
// w_i = base^(-2 i / d_qk), j < d_qk / 4, computed in float64.
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float* table, int max_pos, int quarter, int d_qk, double base) {
  const int64_t n = static_cast<int64_t>(quarter) * max_pos;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(e / max_pos), p = static_cast<int>(e % max_pos);
    float4 out;
    double sn, cs;
    sincos(static_cast<double>(p) * pow(base, -2.0 * (2 * j) / d_qk), &sn, &cs);
    out.x = static_cast<float>(cs);
    out.z = static_cast<float>(sn);
    sincos(static_cast<double>(p) * pow(base, -2.0 * (2 * j + 1) / d_qk), &sn, &cs);
    out.y = static_cast<float>(cs);
    out.w = static_cast<float>(sn);
    reinterpret_cast<float4*>(table)[e] = out;
  }
}

cudaError_t launch_rope_table(float* table, int max_pos, int d_qk, double base, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(d_qk / 4) * max_pos;
  const int blocks = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  rope_table_kernel<<<blocks, 256, 0, s>>>(table, max_pos, d_qk / 4, d_qk, base);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self-test of the failure path: wait on a barrier nothing arrives on.
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(DevStatus st) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, st, KID_SELFTEST);
  __syncthreads();
}

cudaError_t launch_selftest_wait(DevStatus st, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(st);
  return cudaGetLastError();
}

}  // namespace qkvp

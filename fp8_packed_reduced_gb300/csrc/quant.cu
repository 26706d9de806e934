// Bandwidth-bound quantisation kernels:
//   bank refresh  (amax per layer, then codes in both layouts from one pass)
//   x amax        (per-tensor amax of the activations)
//   x quantise    (codes of x, token-major)
//   RoPE table, and the timeout self-test kernel.
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
// partials, then converts a 128 x 128 tile of the bank and writes it to both
// W8 (row-major) and W8T (transposed) from the one read of that tile.  All
// layers of a refresh go in one launch per pass; the second pass reads the
// bank back from L2 for bank sizes that fit there.
// ---------------------------------------------------------------------------
__device__ __forceinline__ const uint16_t* bank_row(const BankArgs& a, int l, int n) {
  if (n < a.Nq) return a.Wq[l] + static_cast<int64_t>(n) * a.D;
  if (n < 2 * a.Nq) return a.Wk[l] + static_cast<int64_t>(n - a.Nq) * a.D;
  return a.Wv[l] + static_cast<int64_t>(n - 2 * a.Nq) * a.D;
}

// grid: (kBankAmaxBlocks, L), 1024 threads.
__global__ void __launch_bounds__(1024) bank_amax_kernel(const __grid_constant__ BankArgs a, float* partials) {
  __shared__ float red[32];
  const int l = blockIdx.y;
  const int row_chunks = a.D / 8;  // 16-byte chunks per row
  const int64_t total = static_cast<int64_t>(a.N) * row_chunks;
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < total; i += 4 * stride) {  // four independent loads in flight
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t e = i + j * stride;
      v[j] = __ldg(reinterpret_cast<const uint4*>(bank_row(a, l, static_cast<int>(e / row_chunks))) +
                   static_cast<int>(e % row_chunks));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, absmax_bf16x8(v[j]));
  }
  for (; i < total; i += stride) {
    const int n = static_cast<int>(i / row_chunks), c = static_cast<int>(i % row_chunks);
    m = fmaxf(m, absmax_bf16x8(__ldg(reinterpret_cast<const uint4*>(bank_row(a, l, n)) + c)));
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) partials[l * gridDim.x + blockIdx.x] = m;
}

// grid: (ceil(N/128) * D/128, L); 256 threads; tile 128 rows x 128 columns.
__global__ void __launch_bounds__(256) bank_quant_kernel(const __grid_constant__ BankArgs a,
                                                         const float* partials) {
  __shared__ float red[32];
  __shared__ __align__(16) uint8_t tr[128][128 + 16];  // [column][row] codes
  const int l = blockIdx.y;
  const int tiles_d = a.D / 128;
  const int n0 = (blockIdx.x / tiles_d) * 128, d0 = (blockIdx.x % tiles_d) * 128;
  const float amax = block_reduce_partials(partials + l * kBankAmaxBlocks, kBankAmaxBlocks, red);
  const float s = scale_from_amax(amax);
  const Bracket k = make_bracket(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) a.w_scale[l] = s;

  const int r = threadIdx.x >> 1;          // tile row
  const int ch = (threadIdx.x & 1) * 64;   // first of this thread's 64 columns
  const int n = n0 + r;
  uint8_t* W8 = a.W8 + static_cast<int64_t>(l) * a.N * a.D;
  uint8_t* W8T = a.W8T + static_cast<int64_t>(l) * a.N * a.D;
  if (n < a.N) {
    const uint4* src = reinterpret_cast<const uint4*>(bank_row(a, l, n) + d0 + ch);
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldg(src + j);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const uint32_t w[8] = {v[j].x, v[j].y, v[j].z, v[j].w, v[j + 1].x, v[j + 1].y, v[j + 1].z, v[j + 1].w};
      uint32_t c[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        c[q] = quant4_fast(bf16_lo(w[2 * q]), bf16_hi(w[2 * q]), bf16_lo(w[2 * q + 1]), bf16_hi(w[2 * q + 1]), k);
      *reinterpret_cast<uint4*>(W8 + static_cast<int64_t>(n) * a.D + d0 + ch + j * 8) =
          make_uint4(c[0], c[1], c[2], c[3]);
#pragma unroll
      for (int b = 0; b < 16; ++b) tr[ch + j * 8 + b][r] = static_cast<uint8_t>(c[b >> 2] >> (8 * (b & 3)));
    }
  } else {
#pragma unroll 1
    for (int b = 0; b < 64; ++b) tr[ch + b][r] = 0;
  }
  __syncthreads();
  // W8T rows d0..d0+127, columns n0..n0+127 (clipped at N); 16 bytes per step.
  const int nvalid = min(128, a.N - n0);
  for (int i = threadIdx.x; i < 128 * 8; i += 256) {
    const int col = i >> 3, part = (i & 7) * 16;
    if (part < nvalid) {
      const uint4 val = *reinterpret_cast<const uint4*>(&tr[col][part]);
      uint8_t* dst = W8T + static_cast<int64_t>(d0 + col) * a.N + n0 + part;
      if (part + 16 <= nvalid) {
        *reinterpret_cast<uint4*>(dst) = val;
      } else {
        const uint8_t* b = reinterpret_cast<const uint8_t*>(&val);
        for (int q = 0; q < nvalid - part; ++q) dst[q] = b[q];
      }
    }
  }
}

cudaError_t launch_bank_amax(const BankArgs& a, float* partials, cudaStream_t s) {
  bank_amax_kernel<<<dim3(kBankAmaxBlocks, a.L), 1024, 0, s>>>(a, partials);
  return cudaGetLastError();
}

cudaError_t launch_bank_quant(const BankArgs& a, const float* partials, cudaStream_t s) {
  const int tiles = ((a.N + 127) / 128) * (a.D / 128);
  bank_quant_kernel<<<dim3(tiles, a.L), 256, 0, s>>>(a, partials);
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
  static int cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int blocks = dev < 64 ? cache[dev] : 0;
  if (blocks <= 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, x_amax_quant_kernel, kFusedThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    blocks = sms * per_sm < kMaxFusedBlocks ? sms * per_sm : kMaxFusedBlocks;
    if (dev < 64) cache[dev] = blocks;
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

/*
 * qkvp.h - C ABI of the reduced-width packed FP8 QKV projection (sm_103a).
 *
 * The operation is the attention-input projection described in
 *   "96 is enough: shrinking attention's routing vectors", section "The change":
 *       W_packed = concat([W_q, W_k, W_v], dim=out)      (96 + 96 + 128 = 320 cols/head)
 *       qkv      = fp8_matmul(x, W_packed)
 *       q, k, v  = split(qkv, [d_qk, d_qk, d_v])
 *       q, k     = rms_norm(q), rms_norm(k)
 *       q, k     = rope(q), rope(k)
 * and in "Track 1 (1.167 min on 8xH100, -5.15% same-node): Reduced-width QK and
 * packed FP8 attention", section "Changes" (one FP8 operation for packed QKV;
 * row-major and transposed FP8 bank cached once per optimizer update from one
 * weight read; norm, RoPE and layout conversion fused; FP8 backward).
 *
 * Conventions shared by every call
 *   - bf16 tensors are passed as uint16_t bit patterns; FP8 tensors as uint8_t
 *     OCP E4M3FN codes; scales as float32 on the device.
 *   - All tensor pointers are DEVICE pointers, owned by the caller; the
 *     library never allocates device memory.  Pointers to arrays of device
 *     pointers (qkvp_quantize_bank) are HOST arrays.
 *   - Every tensor pointer must be 16-byte aligned and row-major/contiguous in
 *     the layout stated at its argument.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream and never synchronise with the host, except
 *     qkvp_poll_device_status.  Calls may be captured into a CUDA graph; the
 *     first call of each kind on a device sizes its launch grids from device
 *     attribute and occupancy queries (cached afterwards), so make it once
 *     before capturing.
 *   - Arguments are validated on the host before anything is launched; on
 *     failure nothing is launched and a qkvp_status other than QKVP_OK is
 *     returned.  No C++ exception crosses this ABI.
 *   - Errors found on the device (a position outside the RoPE table, a
 *     device-side wait that ran out of time) are recorded in the status word
 *     at the start of the workspace and read back by qkvp_poll_device_status.
 *   - Quantisation: per-tensor scale s = amax / 448 in float32 (s = 1 when
 *     amax == 0); code = round-to-nearest-even(v / s) onto E4M3FN with
 *     float32 IEEE division, saturating to +-448.
 *
 * Shapes: T tokens, D model width (multiple of 128), H heads, d_qk in
 * {64, 96, 128}, d_v = 128, N = H * (2*d_qk + d_v) packed rows.
 */
#ifndef QKVP_H_
#define QKVP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qkvp_status {
    QKVP_OK = 0,
    QKVP_ERR_INVALID_ARGUMENT = 1,   /* null pointer, non-positive size, bad eps/base     */
    QKVP_ERR_UNSUPPORTED = 2,        /* shape outside the supported set (see above)       */
    QKVP_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned                 */
    QKVP_ERR_WORKSPACE_TOO_SMALL = 4,/* ws_bytes below the size the call needs           */
    QKVP_ERR_CUDA = 5,               /* a CUDA runtime/driver call or a launch failed    */
    QKVP_ERR_TIMEOUT = 6,            /* device: a bounded wait expired (status word)     */
    QKVP_ERR_DEVICE_INPUT = 7        /* device: a position outside [0, max_pos)          */
} qkvp_status;

typedef struct qkvp_dims {
    int T;      /* tokens (rows of x), 1 .. 2^24                 */
    int D;      /* model width, multiple of 128, 128 .. 16384   */
    int H;      /* heads, 1 .. 128                               */
    int d_qk;   /* Q/K head width: 64, 96 or 128                 */
    int d_v;    /* V head width: 128                             */
} qkvp_dims;

/* Human-readable name of a qkvp_status value (static string, never NULL). */
const char* qkvp_status_string(int status);

/* Bytes of scratch that qkvp_forward and qkvp_backward need for `dims`
 * (one workspace serves both).  0 if dims are unsupported.  The workspace
 * starts with the device status word and the activation quantiser's grid
 * barrier, which every call leaves ready for the next; zero it once with
 * qkvp_workspace_init before first use, and again after a device error (a
 * call that stopped early may leave the barrier mid-count).  It also holds
 * the amax partials, the dW GEMM's split partials and the backward's
 * per-row means of the q/k gradients (2 * H * T floats, written by the dY amax
 * pass and read by the quantise pass).  Calls sharing one workspace must not
 * overlap on the GPU. */
size_t qkvp_workspace_bytes(const qkvp_dims* dims);

/* Bytes of scratch that qkvp_quantize_bank needs for L layers (0 if the
 * shape is unsupported).  The scratch holds the status word and the
 * counters the refresh kernel's blocks share; zero it once with
 * qkvp_workspace_init before first use (every refresh leaves it zeroed),
 * and again after a device error.  Refreshes sharing one scratch must not
 * overlap on the GPU. */
size_t qkvp_bank_workspace_bytes(int L, int D, int H, int d_qk, int d_v);

/* Zero a workspace (status word, grid barrier and all partial buffers).
 * ws: device. */
int qkvp_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Read and clear the device status word at the start of `ws`.  Synchronises
 * `stream`.  Returns QKVP_OK, QKVP_ERR_TIMEOUT or QKVP_ERR_DEVICE_INPUT (the
 * first error recorded since the last poll), or QKVP_ERR_CUDA if the copy
 * failed.  If `where` is non-NULL it receives the id of the kernel that
 * recorded the error (0 when none). */
int qkvp_poll_device_status(void* ws, int* where, void* stream);

/* RoPE table, two rotation pairs per 16-byte entry:
 *   table[(j * max_pos + p) * 4 + {0, 1, 2, 3}]
 *     = cos(p w_2j), cos(p w_2j+1), sin(p w_2j), sin(p w_2j+1),
 * w_i = base^(-2 i / d_qk), j < d_qk/4, 0 <= p < max_pos, computed in float64
 * on the device and stored as float32 ("96 is enough", section "The change":
 * q, k = rope(q), rope(k); rotate-half form).
 *   table: device, 16-byte aligned, d_qk/4 * max_pos * 4 floats. */
int qkvp_build_rope_table(float* table, int max_pos, int d_qk, double base, void* stream);

/* Bank refresh, once per optimizer update ("Track 1 ... packed FP8 attention",
 * section "Changes": row-major and transposed FP8 weight layouts emitted from
 * a single weight read; the logical Q/K/V packs are quantised without
 * materialising their concatenation).
 *   L            layers (1..128)
 *   Wq, Wk, Wv   HOST arrays of L device pointers to bf16 [H*d_qk, D],
 *                [H*d_qk, D], [H*d_v, D] (row-major, out x in)
 *   W8           out, device, [L, N, D] codes; row n of layer l is row n of
 *                concat(W_q, W_k, W_v)
 *   W8T          out, device, [L, D, N] codes, W8T[l] = transpose(W8[l])
 *   w_scale      out, device, [L] float32, one scale per layer (whole bank)
 *   ws           device scratch of qkvp_bank_workspace_bytes(...) bytes,
 *                zeroed once (see qkvp_bank_workspace_bytes)
 * One launch: blocks claim work items (the amax of a 128 x 128 tile, then
 * the codes of a tile) in order from a counter in ws, so the launch needs no
 * particular number of resident blocks and may run beside any other kernel;
 * the code items of a layer wait (bounded, QKVP_ERR_TIMEOUT in the status
 * word) until its amax items are done.  The second read of a tile comes from
 * L2 for banks that fit there, so HBM sees one read of the weights. */
int qkvp_quantize_bank(int L, int D, int H, int d_qk, int d_v,
                       const uint16_t* const* Wq, const uint16_t* const* Wk,
                       const uint16_t* const* Wv,
                       uint8_t* W8, uint8_t* W8T, float* w_scale,
                       void* ws, size_t ws_bytes, void* stream);

/* Bank refresh that allocates nothing, for callers that cannot allocate
 * device memory (no cudaMalloc of their own, no workspace to hand over: for
 * example code confined to a framework's memory pool, or a refresh issued
 * where an allocation could block).  The pages have no counterpart: this is a
 * variant of qkvp_quantize_bank whose scratch (a status word, the counters
 * and per-layer maxima its blocks share) lives in a fixed 2 KB array of
 * device memory inside this library, held by every GPU that loads the
 * library until the process exits.
 *   Arguments and results: as qkvp_quantize_bank, without ws/ws_bytes; bad
 *   arguments give the same status as there.
 *   L above 128 is rejected with QKVP_ERR_UNSUPPORTED (the array's capacity).
 *   The first call in a device's context looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and again after the
 *   context was re-created; make that first call before any stream capture.
 *   Every call shares the one array and clears its status word and counters
 *   (cudaMemsetAsync on `stream`) before its kernel, so nothing is left over
 *   from the previous call.  Calls whose kernels overlap on the GPU
 *   (different streams, or different host threads) race on it: serialise
 *   them.  A device-side wait that runs out (QKVP_ERR_TIMEOUT) is recorded
 *   in the array's own status word, which no poll reads: the refresh's wait
 *   depends only on blocks that are already running. */
int qkvp_quantize_bank_static(int L, int D, int H, int d_qk, int d_v,
                              const uint16_t* const* Wq, const uint16_t* const* Wk,
                              const uint16_t* const* Wv,
                              uint8_t* W8, uint8_t* W8T, float* w_scale, void* stream);

/* Forward ("96 is enough", section "The change"): x is quantised with its own
 * scale, one FP8 GEMM x8 . W8^T (fp32 accumulate) gives the packed columns,
 * and its epilogue de-quantises, splits, RMS-normalises q and k per head
 * (eps inside the square root, no gain), applies rotate-half RoPE at pos[t]
 * and writes head-major bf16.
 *   x         in  [T, D] bf16
 *   pos       in  [T] int32, position of each token inside its sequence
 *   rope_table,max_pos  from qkvp_build_rope_table(d_qk)
 *   W8,w_scale in  one layer of qkvp_quantize_bank: [N, D] codes, [1] float
 *   q, k      out [H, T, d_qk] bf16
 *   v         out [H, T, d_v] bf16
 *   rstd      out [2, H, T] float32: 1/sqrt(mean(Y^2)+eps) of q (0) and k (1)
 *   x8        out [T, D] codes: the GEMM operand, saved for the dW GEMM of
 *               the backward (which reads it token-major, MN-major operand)
 *   x_scale   out [1] float32
 *   ws        scratch, qkvp_workspace_bytes(dims) bytes                    */
int qkvp_forward(const qkvp_dims* dims, float eps,
                 const float* rope_table, int max_pos,
                 const uint16_t* x, const int32_t* pos,
                 const uint8_t* W8, const float* w_scale,
                 uint16_t* q, uint16_t* k, uint16_t* v, float* rstd,
                 uint8_t* x8, float* x_scale,
                 void* ws, size_t ws_bytes, void* stream);

/* The two halves of qkvp_forward as separate calls, so that independent work
 * (for example the bank refresh, on another stream) can run while x is
 * quantised, before the GEMM that needs both.
 *
 * Per-tensor quantisation of any bf16 activation: scale s = amax/448 and
 * codes E(v / s), in one launch (amax, a grid-wide barrier, codes).
 *   x        in  n bf16 values (n a multiple of 16)
 *   x8       out n codes          x_scale out [1] float32
 *   ws       scratch of qkvp_activation_workspace_bytes() bytes, or the
 *            workspace of a forward/backward (its start serves); zeroed
 *            once with qkvp_workspace_init.  Calls sharing it must not
 *            overlap on the GPU.
 * The launch is persistent (two 512-thread blocks per SM, at most 48
 * registers a thread, which leaves a quarter of each SM's registers to other
 * kernels) and its blocks meet at a grid-wide barrier, so all of them must be
 * resident at once: it may share the GPU with small kernels of other streams
 * (the bank refresh, for one), but two of these quantisations (this call, or the one
 * inside qkvp_forward / qkvp_oproj_* / qkvp_mlp_*) running concurrently on
 * different streams, or a long persistent kernel holding the SMs, can keep
 * blocks out until the wait limit (qkvp_set_wait_timeout_ns) expires; the
 * call then reports QKVP_ERR_TIMEOUT through the status word instead of
 * hanging.  Run such calls on one stream. */
size_t qkvp_activation_workspace_bytes(void);
int qkvp_quantize_activation(const uint16_t* x, int64_t n, uint8_t* x8, float* x_scale,
                             void* ws, size_t ws_bytes, void* stream);

/* The forward's packed GEMM and fused epilogue from x8 and x_scale already
 * computed (by qkvp_quantize_activation on x [T, D]); the other arguments
 * and results as in qkvp_forward.  qkvp_forward = qkvp_quantize_activation +
 * qkvp_forward_quantized, with identical results. */
int qkvp_forward_quantized(const qkvp_dims* dims, float eps,
                           const float* rope_table, int max_pos,
                           const uint8_t* x8, const float* x_scale, const int32_t* pos,
                           const uint8_t* W8, const float* w_scale,
                           uint16_t* q, uint16_t* k, uint16_t* v, float* rstd,
                           void* ws, size_t ws_bytes, void* stream);

/* Backward of the forward above ("Track 1 ... packed FP8 attention", sections
 * "Changes" and "Speed": FP8 backward using the cached transposed bank).
 * y is rebuilt from the saved outputs, y = RoPE^T(q), and
 * dY_q = rstd * RoPE^T(dq - q * mean(dq * q)) (the same for k), dY_v = dv;
 * dY is quantised with its own scale into dY8, then
 *   dx = (dY8 . W8) * s_dy * s_w   with the cached W8T as the K-major operand
 *   dW = (dY8^T . x8) * s_dy * s_x with dY8 and x8 read as MN-major operands,
 *        split over tokens; the split partials (fp32, in ws) are summed in
 *        split order by a kernel of their own, so dW is the same on every run
 *   dq, dk    in  [H, T, d_qk] bf16     dv in [H, T, d_v] bf16
 *   q, k      in  [H, T, d_qk] bf16 saved forward outputs
 *   rstd      in  [2, H, T] float32 saved forward output
 *   W8T       in  [D, N] codes of the layer, w_scale [1]
 *   x8        in  [T, D] codes from the forward, x_scale [1]
 *   dx        out [T, D] bf16           dW out [N, D] bf16 (overwritten)
 *   dY8       out [T, N] codes          dy_scale out [1] float32
 *   ws        scratch, qkvp_workspace_bytes(dims) bytes                    */
int qkvp_backward(const qkvp_dims* dims,
                  const float* rope_table, int max_pos,
                  const uint16_t* dq, const uint16_t* dk, const uint16_t* dv,
                  const uint16_t* q, const uint16_t* k, const float* rstd,
                  const int32_t* pos,
                  const uint8_t* W8T, const float* w_scale,
                  const uint8_t* x8, const float* x_scale,
                  uint16_t* dx, uint16_t* dW,
                  uint8_t* dY8, float* dy_scale,
                  void* ws, size_t ws_bytes, void* stream);

/* Diagnostic: launch one kernel that waits on a device barrier nothing ever
 * arrives on, with a wait limit of `timeout_us` microseconds (1..10^6).  The
 * wait expires, the kernel records QKVP_ERR_TIMEOUT in the status word of
 * `ws` and returns; the CUDA context stays usable.  Used to test the
 * failure-reporting path without faulting a GPU. */
int qkvp_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned timeout_us, void* stream);

/* Device-side wait limit used by every kernel (default 2 s, 1 ms .. 60 s). */
int qkvp_set_wait_timeout_ns(uint64_t ns);

/* Kernel timing hook.  Arms `n` (<= 256) caller-created cudaEvent_t handles
 * (HOST array, not copied beyond the handles themselves).  While armed, the
 * calls above record the next unused event on their stream before their
 * first kernel and after each kernel (as external event nodes when the stream
 * is being captured into a CUDA graph), so consecutive events bracket one
 * kernel each.  Order of the kernels: qkvp_quantize_bank: amax, quantise;
 * qkvp_forward: x amax + quantise (one kernel), forward GEMM; qkvp_backward: dY amax,
 * dY quantise, dX GEMM, dW GEMM and its split reduction (two kernels, one
 * interval).  n = 0 disarms.  Not
 * thread-safe; meant for benchmarks. */
int qkvp_set_timing_events(void* const* events, int n);

/* Number of events recorded since the last qkvp_set_timing_events. */
int qkvp_timing_events_recorded(void);

/* GEMM tiling: which of the three GEMMs run on CTA pairs.  Bit 0 = forward,
 * bit 1 = dX, bit 2 = dW.  A paired GEMM computes each 256-row accumulator
 * tile with one tcgen05 MMA over two SMs (a 2-CTA cluster, cta_group::2):
 * each SM loads its own 128 rows of A and half of B, so the shared-memory and
 * L2 traffic of B per SM is halved.  Results are the same either way (every
 * output element is the same fp32 sum over K in the same order).  The dW GEMM
 * is paired only when D is a multiple of 256.  Returns the previous mask, or
 * -1 (mask unchanged) for a mask outside 0..7.  Process-wide, not
 * thread-safe; meant for tests and tuning.  Default 6 (dX and dW paired). */
int qkvp_set_cta_pairs(int mask);

/* ------------------------------------------------------------------------
 * Output projection over the V/O bank ("Track 1 ... packed FP8 attention",
 * section "Changes": Q/K are stored apart from the rectangular V/O bank; FP8
 * weight layouts cached once per optimizer update from one read).  The step
 * after attention: out = a . W_o^T, with a [T, K] the heads' outputs side by
 * side (K = H * d_v) and W_o [D, K] (out x in).  Same FP8 recipe as the
 * packed projection: per-tensor E4M3 scales amax/448 for a, W_o and dout.
 * Shapes: T 1 .. 2^24; D and K multiples of 128, at most 16384.
 * ------------------------------------------------------------------------ */

/* Bytes of scratch qkvp_quantize_weight needs for L matrices [R, C] (0 if
 * unsupported: R, C multiples of 128, R <= 65536, C <= 16384, L <= 128).
 * Zero it once with qkvp_workspace_init (every refresh leaves it zeroed). */
size_t qkvp_weight_workspace_bytes(int L, int R, int C);

/* Refresh of L weight matrices, once per optimizer update: one scale per
 * matrix and its codes in both layouts from one read of the weight.
 *   W      HOST array of L device pointers to bf16 [R, C] (row-major)
 *   W8     out, device, [L, R, C] codes      W8T out, device, [L, C, R] codes
 *   w_scale out, device, [L] float32
 *   ws     device scratch of qkvp_weight_workspace_bytes(L, R, C) bytes      */
int qkvp_quantize_weight(int L, int R, int C, const uint16_t* const* W,
                         uint8_t* W8, uint8_t* W8T, float* w_scale,
                         void* ws, size_t ws_bytes, void* stream);

/* Bytes of scratch qkvp_oproj_forward / qkvp_oproj_backward need (one
 * workspace serves both; zero it once with qkvp_workspace_init, and again
 * after a device error).  0 if the shape is unsupported. */
size_t qkvp_oproj_workspace_bytes(int T, int D, int K);

/* Forward: a is quantised with its own scale, then
 *   out = (a8 . Wo8^T) * s_a * s_o     (one FP8 GEMM, fp32 accumulate)
 *   a        in  [T, K] bf16           Wo8 in [D, K] codes, wo_scale [1]
 *   out      out [T, D] bf16
 *   a8       out [T, K] codes (saved for the backward), a_scale out [1]  */
int qkvp_oproj_forward(int T, int D, int K, const uint16_t* a,
                       const uint8_t* Wo8, const float* wo_scale,
                       uint16_t* out, uint8_t* a8, float* a_scale,
                       void* ws, size_t ws_bytes, void* stream);

/* Backward: dout is quantised with its own scale into dout8, then
 *   da  = (dout8 . Wo8) * s_g * s_o    with the cached Wo8T as the K-major operand
 *   dWo = (dout8^T . a8) * s_g * s_a   split over tokens, reduced in split
 *                                      order inside the GEMM (deterministic)
 *   dout     in  [T, D] bf16           Wo8T in [K, D] codes, wo_scale [1]
 *   a8       in  [T, K] codes from the forward, a_scale [1]
 *   da       out [T, K] bf16           dWo out [D, K] bf16 (overwritten)
 *   dout8    out [T, D] codes          dout_scale out [1] float32           */
int qkvp_oproj_backward(int T, int D, int K, const uint16_t* dout,
                        const uint8_t* Wo8T, const float* wo_scale,
                        const uint8_t* a8, const float* a_scale,
                        uint16_t* da, uint16_t* dWo,
                        uint8_t* dout8, float* dout_scale,
                        void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * FP8 ReLU-squared MLP ("Track 1 ... packed FP8 attention", section
 * "Changes": FP8 across the whole ReLU-squared forward and backward path and
 * all of its GEMMs; the saved pre-activation is dropped, relu(pre) being
 * recoverable from the stored squared activation):
 *   h = relu(x . W_fc^T)^2,  out = h . W_proj^T
 * with W_fc [F, D] and W_proj [D, F] (out x in), F the hidden width.  Weights
 * are refreshed by qkvp_quantize_weight (both layouts).  Per-tensor E4M3
 * scales amax/448 for x, h, dout and dpre.  h and dpre are produced in bf16
 * by the GEMM that makes them (which also reduces their amax) and quantised
 * from there; the backward rebuilds relu(pre) = sqrt(h^) from the stored
 * codes h8.  Shapes: T 1 .. 2^24; D a multiple of 128 up to 16384; F a
 * multiple of 128 up to 65536.
 * ------------------------------------------------------------------------ */

/* Bytes of scratch qkvp_mlp_forward / qkvp_mlp_backward need (one workspace
 * serves both; zero it once with qkvp_workspace_init, and again after a
 * device error).  0 if the shape is unsupported. */
size_t qkvp_mlp_workspace_bytes(int T, int D, int F);

/* Forward:
 *   x        in  [T, D] bf16
 *   W1_8     in  [F, D] codes of W_fc, w1_scale [1]
 *   W2_8     in  [D, F] codes of W_proj, w2_scale [1]
 *   out      out [T, D] bf16
 *   x8       out [T, D] codes, x_scale [1]           (saved for the backward)
 *   h        out [T, F] bf16 squared activation (an intermediate; may be
 *                reused by the caller once the call has run, e.g. as dpre)
 *   h8       out [T, F] codes, h_scale [1]           (saved for the backward) */
int qkvp_mlp_forward(int T, int D, int F, const uint16_t* x,
                     const uint8_t* W1_8, const float* w1_scale,
                     const uint8_t* W2_8, const float* w2_scale,
                     uint16_t* out, uint8_t* x8, float* x_scale,
                     uint16_t* h, uint8_t* h8, float* h_scale,
                     void* ws, size_t ws_bytes, void* stream);

/* Backward:
 *   dout     in  [T, D] bf16
 *   W1_8T    in  [D, F] codes (W_fc transposed), w1_scale [1]
 *   W2_8T    in  [F, D] codes (W_proj transposed), w2_scale [1]
 *   x8, h8   in  the forward's saved codes and scales
 *   dx       out [T, D] bf16      = dpre^ . W_fc^
 *   dW1      out [F, D] bf16      = dpre^^T . x^   (split over tokens, fixed order)
 *   dW2      out [D, F] bf16      = dout^^T . h^   (split over tokens, fixed order)
 *   dout8    out [T, D] codes, dout_scale [1]
 *   dpre     out [T, F] bf16      = (dout^ . W_proj^) * 2 sqrt(h^) (intermediate)
 *   dpre8    out [T, F] codes, dpre_scale [1]                              */
int qkvp_mlp_backward(int T, int D, int F, const uint16_t* dout,
                      const uint8_t* W1_8T, const float* w1_scale,
                      const uint8_t* W2_8T, const float* w2_scale,
                      const uint8_t* x8, const float* x_scale,
                      const uint8_t* h8, const float* h_scale,
                      uint16_t* dx, uint16_t* dW1, uint16_t* dW2,
                      uint8_t* dout8, float* dout_scale,
                      uint16_t* dpre, uint8_t* dpre8, float* dpre_scale,
                      void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QKVP_H_ */

/*
 * w4a8.h -- C ABI of the GB300 weight-quantized decode linear library.
 *
 * The method (pages it follows):
 *  - "Jetson Orin AGX 上的 INT4 量化推理实践：从 9 tok/s 到 19.6 tok/s",
 *    sections 当前实现方式 and 正确方向: weights quantized row-wise to INT4
 *    with one scale per output row; the activation quantized dynamically to
 *    INT8 before every linear; int8 x int8 products accumulated in int32;
 *    output = int32 accumulate * weight_scale * activation_scale, as float.
 *    Section 后续优化方向 lists the fusion of the activation quantization
 *    into the linear kernel (w4a8_linear below).
 *  - "TPU-MLIR W8A16 for ChatGLM2-6B", sections 2-4: per-channel INT8
 *    weights, cast back to floating point and multiplied by the scale, then
 *    multiplied with the F16 activation (w8a16_gemv below).
 *  - "IntAttention" (MLSys 2026), section 基准/方法设计: the IndexSoftmax
 *    integer softmax (index_softmax_u8 below).
 *
 * Readings of points the pages leave open (fixed here, identical in the
 * CPU oracle used by the tests):
 *  - INT4 codes are symmetric in [-7, 7]: s_w = max|w_row| / 7 (fp32 IEEE
 *    division), q = clamp(round_half_away(w / s_w), -7, 7).
 *  - INT8 activation codes are in [-127, 127]: s_a = max|x_row| / 127,
 *    q = clamp(round_half_away(x / s_a), -127, 127); one s_a per activation
 *    row.  A zero row gets scale 0 and all codes 0.
 *  - Packing: byte j of a weight row holds code 2j in bits 0..3 and code
 *    2j+1 in bits 4..7, each a 4-bit two's-complement value.
 *  - Rescale: Y = ((float)acc * s_w) * s_a, two fp32 round-to-nearest
 *    multiplies in that order.  W4A8 results are therefore exact functions
 *    of the inputs (bit-reproducible).
 *  - W8A16: s = binary16(max|w_row| / 127) per output channel; codes are
 *    taken with that rounded scale; Y = s * sum_k float(q) * float(x) with
 *    fp32 accumulation (order unspecified; within a stated tolerance of the
 *    fp64 result).
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers owned by the caller, row-major
 *    and contiguous.  binary16 data is passed as uint16_t bit patterns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous on that stream and performs no
 *    host synchronisation and no allocation.
 *  - Arguments are checked on the host before any launch; a failed check
 *    returns a W4A8_ERR_* code, launches nothing and leaves a message for
 *    w4a8_last_error().  A launch failure returns W4A8_ERR_CUDA.
 *  - Inputs must be finite; results for NaN or Inf inputs are unspecified.
 *  - No kernel traps.  Device-side waits are bounded (about 2 s); a wait that
 *    runs out sets a bit in a device error word (see w4a8_device_error) and
 *    the kernel returns early with its outputs unspecified.
 */
#ifndef W4A8_H
#define W4A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A8_OK = 0,
    W4A8_ERR_NULL = 1,      /* a required pointer is NULL */
    W4A8_ERR_ALIGN = 2,     /* a pointer is not aligned as documented */
    W4A8_ERR_SHAPE = 3,     /* a size is out of the documented range */
    W4A8_ERR_WORKSPACE = 4, /* workspace missing or smaller than required */
    W4A8_ERR_CUDA = 5       /* a CUDA call failed (message has the reason) */
} w4a8_status_t;

/* Launch flag: allow the kernel to start while the previous kernel on the
   stream is still running (programmatic dependent launch).  The kernel then
   streams Wq/Wq8 and the weight scales before waiting for the previous
   kernel, so those weight buffers must NOT be written by the kernel launched
   immediately before it on the same stream.  Activations, outputs and the
   workspace are only touched after the wait. */
#define W4A8_LAUNCH_PDL 1u

/* Maximum activation rows (decode batch) per call.  Which kernel serves a
 * call (w4a8_plan_info reports it; w4a8_tuning_t moves the thresholds):
 *  - 1 row: the dp4a GEMV (fused activation quantization, weights streamed
 *    by bulk copies into a shared-memory ring).
 *  - row-wise scales, 2 or 3 rows on matrices of at most 2 x SMs 128-row
 *    tiles: the row-per-thread integer kernel (an activation pass writes the
 *    codes split by parity; four threads of four warps walk each weight row,
 *    unpack its INT4 codes once for all batch rows and sum exact int32 dp4a
 *    products against shared-memory broadcasts of the activations).
 *  - other row-wise calls from 2 rows: the tcgen05 tensor cores.  An
 *    activation pass writes each INT8 code as two exact e4m3 integers
 *    (a = 16 a_hi + a_lo); converter warps turn each INT4 code into the e4m3
 *    byte q + 8, which is exactly (q + 8) * 2^-9, and store it into TMEM;
 *    kind::f8f6f4 MMAs of 128 weight rows x 32 codes x the batch accumulate
 *    exactly in fp32 (every partial sum of one K piece of at most 16384 is
 *    an integer multiple of 2^-9 below 2^15), and the bias 8 * sum(a) is
 *    removed with the exact code sum, so the rescale matches the dp4a path
 *    bit for bit.
 *  - group-wise scales: the one-thread-per-row integer kernel for 1..8 rows
 *    (each thread folds its weight row's group sums in the fixed order of
 *    the group-scale contract), the tensor cores (binary16 operands) from 9
 *    rows for groups of whole 128-code stages up to 16384 codes, otherwise
 *    the one-thread-per-row kernel once per group of up to 8 rows.
 *  - the warp-level e4m3 MMA kernel (mma.sync m16n8k32, operands built in
 *    registers) serves row-wise calls of 2..4 rows on matrices of at least
 *    4 x SMs 128-row tiles in one K piece (lm_head-sized: persistent CTAs,
 *    two per SM, walk the tiles), ahead of the tensor cores; and 2..32 rows
 *    on any matrix when w4a8_tuning_t.qmma_max_m asks for it.
 * When the other kernels are switched off the dp4a GEMV serves batches too,
 * one launch per group of up to 8 rows (W8A16: always, 4 rows, fp32 FMAs),
 * each streaming the whole weight matrix.  w4a8_linear_noalloc takes at most
 * 8 rows, on the kernel above whose workspace fits its static scratch, else
 * on the dp4a GEMV in one launch. */
#define W4A8_MAX_M 64
#define W8A16_MAX_M 64

/* ---------------------------------------------------------------------- */
/* Weight quantizers (load time)                                           */
/* ---------------------------------------------------------------------- */

/* Row-wise INT4 weight quantization and packing (the Jetson INT4 page,
 * section 当前实现方式: "row-wise INT4 packed weight, one scale per row").
 *   W   [N][K] fp32 in;  Wq [N][K/2] uint8 out;  sw [N] fp32 out.
 *   Requires N >= 1, K >= 32, K % 32 == 0; W and Wq 16-byte aligned.
 * Bit-identical to the CPU definition for finite inputs. */
int w4_quantize_weights(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* sw,
                        void* stream);

/* Per-output-channel INT8 weight quantization (the TPU-MLIR W8A16 page,
 * section 2: per-channel INT8 storage; section 3: F16 scales).
 *   W [N][K] fp32 in;  Wq8 [N][K] int8 out;  sw16 [N] binary16 out.
 *   Requires N >= 1, K >= 16, K % 16 == 0; W and Wq8 16-byte aligned. */
int w8_quantize_weights(const float* W, int64_t N, int64_t K, int8_t* Wq8, uint16_t* sw16,
                        void* stream);

/* ---------------------------------------------------------------------- */
/* Activation quantizer                                                    */
/* ---------------------------------------------------------------------- */

/* Dynamic INT8 activation quantization, one scale per row (the Jetson INT4
 * page, section 正确方向: "activation: dynamically quantized to INT8").
 *   X [M][K] binary16 in;  Xq [M][K] int8 out;  sa [M] fp32 out.
 *   Requires 1 <= M <= 65535, 1 <= K <= 2^20, K % 8 == 0; X and Xq 16-byte
 *   aligned. */
int act_quantize_i8(const uint16_t* X, int64_t M, int64_t K, int8_t* Xq, float* sa,
                    void* stream);

/* ---------------------------------------------------------------------- */
/* W4A8 linear                                                             */
/* ---------------------------------------------------------------------- */

/* Workspace bytes w4a8_gemv / w4a8_linear need for this shape on the
 * current device (0 when the chosen plan does not split K).  Layout: 4096
 * bytes of arrival counters, then scratch (split partials; for the
 * tensor-core path the activation codes and int32 accumulators, which its
 * first kernel clears).  The counters must be zero before the first call
 * (zero-fill the buffer once); every call leaves them zero, so one
 * workspace can serve calls of any shape, in either precision (after a
 * non-zero w4a8_device_error, zero-fill it again).  Calls that share a workspace must not run
 * concurrently (same stream, or ordered by events).  Returns 0 for shapes
 * the linear entry points reject. */
size_t w4a8_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* INT4-weight x INT8-activation product with int32 accumulation and fp32
 * rescale (the Jetson INT4 page, sections 正确方向 and 当前实现方式).
 *   Xq [M][K] int8, sa [M] fp32      quantized activation (act_quantize_i8)
 *   Wq [N][K/2] uint8, sw [N] fp32   packed weights (w4_quantize_weights)
 *   Y  [M][N] fp32 out: Y[m][n] = ((float)acc[m][n] * sw[n]) * sa[m]
 *   acc_out [M][N] int32 out, optional (NULL to skip): the exact
 *     acc[m][n] = sum_k Xq[m][k] * q[n][k]
 *   ws, ws_bytes: workspace of at least w4a8_workspace_bytes(M, K, N)
 *     bytes, 256-byte aligned (may be NULL when that is 0).
 *   flags: 0 or W4A8_LAUNCH_PDL.
 * Requires 1 <= M <= W4A8_MAX_M, 32 <= K <= 131072, K % 32 == 0,
 * 1 <= N <= 2^31 - 1; Xq and Wq 16-byte aligned; Y, sw, sa 4-byte aligned. */
int w4a8_gemv(const int8_t* Xq, const float* sa, int64_t M, int64_t K, const uint8_t* Wq,
              const float* sw, int64_t N, float* Y, int32_t* acc_out, void* ws,
              size_t ws_bytes, unsigned flags, void* stream);

/* Fused linear: activation quantization + INT4 x INT8 product + rescale in
 * one kernel (the Jetson INT4 page, section 后续优化方向: fold the
 * activation quantize into the linear kernel and save a launch).
 *   X [M][K] binary16 in; Wq, sw, Y, acc_out, ws, ws_bytes, flags as in
 *   w4a8_gemv.  Xq_out [M][K] int8 and sa_out [M] fp32 are optional outputs
 *   (NULL to skip) holding exactly what act_quantize_i8 would produce.
 * Y is bit-identical to act_quantize_i8 followed by w4a8_gemv.
 * Requires the w4a8_gemv shape limits; X 16-byte aligned. */
int w4a8_linear(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const float* sw,
                int64_t N, float* Y, int8_t* Xq_out, float* sa_out, int32_t* acc_out,
                void* ws, size_t ws_bytes, unsigned flags, void* stream);

/* Grouped fused linear: G weight matrices that read the same activation
 * (the query/key/value projections, or the gate and up projections of an
 * MLP) in one launch, quantizing the activation once (the Jetson INT4 page,
 * section 后续优化方向: cut the repeated quantization in QKV and the MLP).
 *   X [M][K] binary16 in;  for g < G: Wq[g] [N[g]][K/2] uint8, sw[g] [N[g]]
 *   fp32, Y[g] [M][N[g]] fp32 out; Wq, sw, N, Y are HOST arrays of G device
 *   pointers / sizes.  Y[g] is bit-identical to w4a8_linear(X, Wq[g], sw[g]).
 *   ws, ws_bytes: at least w4a8_workspace_bytes(M, K, N[0] + ... + N[G-1]).
 * Requires 1 <= G <= W4A8_MAX_GROUP and the w4a8_linear limits with
 * N = the sum of N[g]; X and every Wq[g] 16-byte aligned. */
#define W4A8_MAX_GROUP 4
int w4a8_linear_grouped(const uint16_t* X, int64_t M, int64_t K, int G, const uint8_t* const* Wq,
                        const float* const* sw, const int64_t* N, float* const* Y, void* ws,
                        size_t ws_bytes, unsigned flags, void* stream);

/* Fused linear that allocates nothing and takes no workspace.  The pages
 * have no counterpart; this is a calling convention for callers that cannot
 * provide device memory: code paths that must not allocate, such as an
 * engine's per-token execute step or a framework plugin whose enqueue
 * function is not allowed to, because cudaMalloc can synchronise the device
 * and take unbounded time.
 *   Same arguments and results as w4a8_linear without the optional outputs,
 *   for 1 <= M <= 8: Y is bit-identical to w4a8_linear's.  The call runs the
 *   kernel w4a8_linear would (the routing above) when that plan's workspace
 *   fits the static scratch, else the dp4a GEMV in one launch.
 * The scratch is a static 4 MiB device array (W4A8_NOALLOC_SCRATCH bytes:
 * 4096 bytes of arrival counters, then the kernels' workspace) that every GPU
 * loading the library holds until the process exits.  Shapes whose dp4a plan
 * also needs more scratch are rejected with W4A8_ERR_WORKSPACE (at M = 1 and
 * four K pieces that is N > 261,888).  Each call that needs scratch looks up the
 * array's device address on the current device (a lookup, no allocation);
 * the first call on a device may load the library's device code there, so
 * make it before any stream capture.  Every call on a device shares the one
 * array, which keeps the last call's contents; the array starts zeroed and
 * the kernels leave its counters at zero, so calls in order on one stream
 * are fine, but calls whose executions overlap on the GPU (different
 * streams without ordering between them) race and give wrong results.  A
 * call whose kernel gave up on a bounded wait may leave the counters
 * non-zero; w4a8_device_error, which reports that, also clears them. */
#define W4A8_NOALLOC_SCRATCH (4u << 20)
int w4a8_linear_noalloc(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                        const float* sw, int64_t N, float* Y, unsigned flags, void* stream);

/* ---------------------------------------------------------------------- */
/* The MLP's gated product: gate/up projections -> down projection          */
/* ---------------------------------------------------------------------- */

/* The INT4 page's model (HIDDEN 3584, INTERMEDIATE 18944) has the MLP
 * down(silu(gate(x)) * up(x)); section 后续优化方向 asks to cut the
 * quantization overhead of the MLP.  The page does not print the
 * activation; the reading is that model family's SwiGLU, silu(g) = g / (1 +
 * exp(-g)).  The calls below produce the down projection's binary16 input h
 * where gate and up are produced, so down (w4a8_linear on h) quantizes one
 * binary16 vector and no separate launch sits between the two linears.
 *
 * Contract, per element: h = binary16(silu(g) * u) computed in fp32 (expf
 * within 2 ulp, then one add, one division, one multiply, each rounded to
 * nearest, then one round-to-nearest-even conversion).  The fp32 value is
 * within 2^-20 |v| of v = silu(g) * u in exact arithmetic, so h equals the
 * binary16 rounding of v unless v lies within 2^-20 |v| of a binary16
 * rounding boundary (where either neighbour may result). */

/* Interleaves the rows of two packed weight matrices of the same shape
 * (gate and up): out row 2i = a row i, out row 2i + 1 = b row i, and the same
 * for the scales.  Quantization is row-wise, so this equals quantizing the
 * row-interleaved fp32 matrix.  Device-to-device copies on `stream`.
 *   Wq_a, Wq_b [N][K/2] uint8, sw_a, sw_b [N] fp32 in;
 *   Wq_out [2N][K/2] uint8, sw_out [2N] fp32 out.
 * Requires 1 <= N <= 2^30 - 1, K >= 32, K % 32 == 0. */
int w4_interleave_rows(const uint8_t* Wq_a, const float* sw_a, const uint8_t* Wq_b, const float* sw_b,
                       int64_t N, int64_t K, uint8_t* Wq_out, float* sw_out, void* stream);

/* Workspace bytes of w4a8_gate_up_silu (rules of w4a8_workspace_bytes). */
size_t w4a8_gate_up_silu_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* Gate and up projections with the gated product in the epilogue.
 *   X [M][K] binary16 in; Wq_gu [2N][K/2], sw_gu [2N]: gate and up
 *   interleaved by rows (w4_interleave_rows);
 *   Y_gu [M][2N] fp32 out: Y_gu[m][2i] = gate i, Y_gu[m][2i+1] = up i, each
 *     bit-identical to w4a8_linear on that projection;
 *   H [M][N] binary16 out: H[m][i] = binary16(silu(Y_gu[m][2i]) *
 *     Y_gu[m][2i+1]) under the contract above;
 *   ws, ws_bytes (w4a8_gate_up_silu_workspace_bytes), flags as w4a8_linear.
 * One row: one launch of the fused GEMV, each CTA owning whole gate/up row
 * pairs and writing their products after its outputs.  Batches of 2+ rows:
 * the W4A8 linear on the interleaved matrix, then the product as a launch of
 * its own (w4a8_silu_mul's kernel).
 * Requires the w4a8_linear limits with 2N output rows; X and Wq_gu 16-byte,
 * Y_gu and sw_gu 4-byte, H 2-byte aligned. */
int w4a8_gate_up_silu(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq_gu, const float* sw_gu,
                      int64_t N, float* Y_gu, uint16_t* H, void* ws, size_t ws_bytes, unsigned flags,
                      void* stream);

/* The gated product on its own (the unfused step):
 *   H[m][i] = binary16(silu(g[m][i]) * u[m][i]), g, u [M][N] fp32,
 *   H [M][N] binary16, same contract.  flags: 0 or W4A8_LAUNCH_PDL.
 * Requires 1 <= M <= 65535, 1 <= N <= 2^31 - 1; g, u 4-byte, H 2-byte
 * aligned. */
int w4a8_silu_mul(const float* g, const float* u, int64_t M, int64_t N, uint16_t* H, unsigned flags,
                  void* stream);

/* Decode-step prefetch (no counterpart on the pages): w4a8_linear and
 * w4a8_linear_grouped with a hint, `next`, `next_bytes`: the first bytes of
 * the weights the following launch will read.  When the call runs the
 * one-row dp4a GEMV, its CTAs bring that range into L2 at the start (a
 * cp.async.bulk.prefetch.L2 of each CTA's share), while the launch, which at
 * one row is bound by latency, leaves HBM idle; the following launch then
 * finds those bytes in L2.  Other kernels ignore the hint.  A hint changes
 * no result.  Requires next 16-byte aligned (NULL = none); next_bytes is
 * rounded down to a multiple of 16. */
int w4a8_linear_prefetch(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const float* sw,
                         int64_t N, float* Y, void* ws, size_t ws_bytes, unsigned flags, void* stream,
                         const void* next, size_t next_bytes);
int w4a8_linear_grouped_prefetch(const uint16_t* X, int64_t M, int64_t K, int G, const uint8_t* const* Wq,
                                 const float* const* sw, const int64_t* N, float* const* Y, void* ws,
                                 size_t ws_bytes, unsigned flags, void* stream, const void* next,
                                 size_t next_bytes);

/* ---------------------------------------------------------------------- */
/* W4A8 with group-wise weight scales                                      */
/* ---------------------------------------------------------------------- */

/* Group-wise scales (the Jetson INT4 page, section 后续优化方向, which names
 * group-wise scales as the next step for precision): one fp32 scale per
 * group of `group` consecutive codes of a weight row instead of one per row.
 * `group` is a power of two from 32 to K that divides K.  Scale rows are
 * padded to 16 bytes: sg is [N][W4G_SCALE_STRIDE(K, group)] fp32, the
 * stride being K/group rounded up to a multiple of 4; w4g_quantize_weights
 * writes the padding entries as 0 and the products never use them. */
#define W4G_SCALE_STRIDE(K, group) ((((K) / (group)) + 3) / 4 * 4)

/* Group-wise INT4 weight quantization: for each row n and group g,
 * s = max|W over the group| / 7 (fp32 IEEE division),
 * q = clamp(round_half_away(w / s), -7, 7), packed as w4_quantize_weights.
 * With group == K the codes and scales are those of w4_quantize_weights.
 *   W [N][K] fp32 in;  Wq [N][K/2] uint8 out;  sg [N][stride] fp32 out.
 *   Requires N >= 1, K >= 32, K % 32 == 0, the group rule above; W, Wq
 *   and sg 16-byte aligned.
 * Bit-identical to the CPU definition for finite inputs. */
int w4g_quantize_weights(const float* W, int64_t N, int64_t K, int64_t group, uint8_t* Wq,
                         float* sg, void* stream);

/* Workspace bytes of w4a8g_gemv / w4a8g_linear (rules of
 * w4a8_workspace_bytes; 0 also for shapes those calls reject). */
size_t w4a8g_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t group);

/* INT4 x INT8 product with group-wise weight scales:
 *   Y[m][n] = sa[m] * sum_g sg[n][g] * acc_g[m][n],
 *   acc_g[m][n] = sum over the codes k of group g of Xq[m][k] * q[n][k].
 * Arithmetic, in an order fixed by K and group alone (the page gives the
 * output as the integer sum times the weight and activation scales, per
 * group, and fixes no summation order):
 *   acc_g is exact (int32; converted to fp32 with one round-to-nearest,
 *     exact for groups of at most 16384 codes);
 *   the fold chunks are L = max(group, 1024) codes: per chunk, f = +0, then
 *     for its groups in ascending order f = fmaf(acc_g, s_g, f) (one
 *     rounding each);
 *   T = +0, then for the chunks in ascending order T = T + f;
 *   Y[m][n] = T * sa[m].
 * So Y is the same bits whatever the batch size, kernel or K split, and
 * lies within (L / group + ceil(K / L) + 1) * 2^-24 * sa[m] * sum_g sg[n][g]
 * * |acc|_g of the exact value, |acc|_g being the sum of |Xq * q| over
 * group g.  Kernels: 1..8 rows (w4a8_tuning_t.rowdot_max_m) one thread per
 * weight row, which walks the row's codes in order (K pieces of whole
 * chunks; with split K each chunk's f goes to the workspace and the CTA that
 * finishes a tile last adds them in chunk order).  From 9 rows
 * (w4a8_tuning_t.mma_min_m) with a group of a multiple of 128 codes up to
 * 16384: the tensor cores, each group's products summed exactly in an fp32
 * TMEM accumulator, the fold run by the epilogue threads (K not split).
 * Other calls: the one-thread-per-row kernel once per group of up to 8 rows.
 *   Xq [M][K] int8, sa [M] fp32    quantized activation (act_quantize_i8)
 *   Wq [N][K/2] uint8, sg [N][stride] fp32   (w4g_quantize_weights)
 *   Y [M][N] fp32 out; ws, ws_bytes (w4a8g_workspace_bytes) and flags as
 *   in w4a8_gemv.
 * Requires 1 <= M <= W4A8_MAX_M, the w4a8_gemv limits on K and N, the group
 * rule above; Xq, Wq and sg 16-byte aligned; Y and sa 4-byte aligned. */
int w4a8g_gemv(const int8_t* Xq, const float* sa, int64_t M, int64_t K, int64_t group,
               const uint8_t* Wq, const float* sg, int64_t N, float* Y, void* ws,
               size_t ws_bytes, unsigned flags, void* stream);

/* Fused linear with group-wise scales: activation quantization and the
 * product above in one kernel.  Xq_out [M][K] int8 and sa_out [M] fp32 are
 * optional outputs (NULL to skip), bit-identical to act_quantize_i8's; Y is
 * bit-identical to act_quantize_i8 followed by w4a8g_gemv.
 * Requires the w4a8g_gemv limits; X 16-byte aligned. */
int w4a8g_linear(const uint16_t* X, int64_t M, int64_t K, int64_t group, const uint8_t* Wq,
                 const float* sg, int64_t N, float* Y, int8_t* Xq_out, float* sa_out, void* ws,
                 size_t ws_bytes, unsigned flags, void* stream);

/* Grouped fused linear with group-wise scales: G weight matrices reading
 * the same activation in one launch, as w4a8_linear_grouped.  Wq, sg, N, Y
 * are HOST arrays of G device pointers / sizes; ws covers
 * w4a8g_workspace_bytes(M, K, N[0] + ... + N[G-1], group).  Y[g] is
 * bit-identical to w4a8g_linear's on matrix g (the order is fixed by K and
 * group, not by the launch plan). */
int w4a8g_linear_grouped(const uint16_t* X, int64_t M, int64_t K, int64_t group, int G,
                         const uint8_t* const* Wq, const float* const* sg, const int64_t* N,
                         float* const* Y, void* ws, size_t ws_bytes, unsigned flags,
                         void* stream);

/* ---------------------------------------------------------------------- */
/* W8A16 linear                                                            */
/* ---------------------------------------------------------------------- */

/* Workspace bytes w8a16_gemv needs (same rules as w4a8_workspace_bytes). */
size_t w8a16_workspace_bytes(int64_t M, int64_t K, int64_t N);

/* INT8-weight x F16-activation product (the TPU-MLIR W8A16 page,
 * section 4: cast INT8 to floating point, multiply by the scale, multiply
 * with the activation).  The code is widened to binary16 exactly in
 * registers, each binary16 x binary16 product is exact in fp32, sums are
 * fp32, and the per-channel scale is applied once per output:
 * Y[m][n] = float(sw16[n]) * sum_k q[n][k]*x[m][k].
 *   X [M][K] binary16, Wq8 [N][K] int8, sw16 [N] binary16, Y [M][N] fp32.
 * Requires 1 <= M <= W8A16_MAX_M, 16 <= K <= 65536, K % 16 == 0,
 * 1 <= N <= 2^31 - 1; X and Wq8 16-byte aligned, Y 4-byte aligned. */
int w8a16_gemv(const uint16_t* X, int64_t M, int64_t K, const int8_t* Wq8,
               const uint16_t* sw16, int64_t N, float* Y, void* ws, size_t ws_bytes,
               unsigned flags, void* stream);

/* ---------------------------------------------------------------------- */
/* IndexSoftmax (integer softmax of attention logits)                      */
/* ---------------------------------------------------------------------- */

/* IndexSoftmax (page "【MLSys 2026】IntAttention：全整数注意力流水线，边缘推理的高效部署",
 * section 基准/方法设计, mechanisms 1-3): int32 attention logits (an INT8 x INT8
 * QK^T product) to UINT8 probabilities without floating point, per row:
 *   delta = rowMax(A) - A;  delta' = min(delta, c_int)
 *   idx   = round(delta' * (2^b - 1) / c_int);  E = LUT[idx]
 *   P     = round(255 * E / rowSum(E))
 * Every rounding takes halves up (all operands are non-negative); c_int = 0
 * clips every distance to 0.  P is bit-identical to the CPU definition. */

/* The page's hyperparameters, b = 5 (a 32-entry table) and c = 6.6. */
#define ISX_DEFAULT_B 5
#define ISX_DEFAULT_C 6.6
#define ISX_MAX_COLS (1 << 23)

/* Host-only (no GPU): fills lut[0 .. 2^b - 1] with
 * LUT[i] = round(255 * exp(-c * i / (2^b - 1))) in binary64, LUT[2^b - 1] = 0.
 * Requires 1 <= b <= 8 and c > 0. */
int index_softmax_lut(int b, double c, uint8_t* lut);

/* Host-only: the clipping threshold in logit units,
 * c_int = round(c * sqrt(d) / (s_q * s_k)) in binary64, for per-tensor INT8
 * scales s_q, s_k and head dimension d.  Returns -1 unless c > 0, d >= 1,
 * s_q > 0, s_k > 0 and the result fits in [0, 2^31 - 1]. */
int64_t index_softmax_c_int(double c, int64_t d, float s_q, float s_k);

/* P[rows][cols] = IndexSoftmax(A[rows][cols]) row by row.
 *   A: int32 logits (device); P: UINT8 probabilities out (device).
 *   c_int: threshold (index_softmax_c_int); b: table bits; lut: HOST array
 *   of 2^b entries (index_softmax_lut, or any table with lut[0] >= 1, which
 *   keeps every row sum positive), copied into the launch.
 * Requires 1 <= rows <= 2^31 - 1, 1 <= cols <= ISX_MAX_COLS,
 * 0 <= c_int <= 2^31 - 1, 1 <= b <= 8, lut[0] >= 1; A 4-byte aligned.
 * cols % 4 == 0 with A 16-byte and P 4-byte aligned takes the vector path;
 * rows of up to 8192 (vector path) or 1024 elements stay in registers (one
 * read of A), longer rows are read three times. */
int index_softmax_u8(const int32_t* A, int64_t rows, int64_t cols, int64_t c_int, int b,
                     const uint8_t* lut, uint8_t* P, void* stream);

/* ---------------------------------------------------------------------- */
/* Diagnostics                                                             */
/* ---------------------------------------------------------------------- */

/* Message for the last non-OK status returned on the calling thread
 * ("" if none).  The pointer stays valid until the next call on this
 * thread. */
const char* w4a8_last_error(void);

/* Copies the current device's error word into *flags and clears it.  Bit 0:
 * a wait for weight data ran out; bit 1: unused; bit 2: a wait for
 * in-flight copies at exit ran out.  A non-zero word means that some call's
 * outputs are unspecified and that the split-K arrival counters of the
 * workspace it used may be left non-zero: zero-fill that workspace again
 * before reusing it.  (The static scratch of w4a8_linear_noalloc is cleared
 * here, on `stream`, whenever the word is non-zero.)
 * Synchronises `stream` first.  Returns W4A8_OK or W4A8_ERR_CUDA. */
int w4a8_device_error(unsigned* flags, void* stream);

/* ---------------------------------------------------------------------- */
/* Tuning and introspection (no counterpart on the pages)                  */
/* ---------------------------------------------------------------------- */

/* Process-wide overrides of the launch plan, for A/B measurements and for
 * tests that must exercise a given plan.  Zero fields keep the heuristic.
 *   force_splits: number of K pieces (1..16); the shape must admit it
 *     (group-wise scales on the one-thread-per-row kernel: pieces of whole
 *     fold chunks, so at most the chunk count, fewer when the chunks do not
 *     divide evenly; tensor cores: never split).
 *   force_threads_per_row: threads sharing one row-piece (power of 2, <=256).
 *   ring_bytes: target size of the shared-memory weight ring (<= 204800).
 *   ctas_per_sm: CTAs per SM for each K piece (1..4; 0 = 1); for the
 *     row-per-thread kernel, CTAs per SM (0 = 1 at 4 or 8 threads per
 *     row, 2 at 2; 4 for the group-scale kernel).
 *   mma_min_m: activation rows from which the W4A8 entry points use the
 *     tensor-core kernel (2..65; 0 = default: 2 rows for row-wise scales,
 *     3 for group-wise scales; 65 = never).
 *   rowdot_max_m: activation rows up to which W4A8 calls use the
 *     row-per-thread kernel in one launch, from 2 rows (group-wise scales:
 *     from 1) (0 = default: 3 rows for row-wise scales on matrices of at
 *     most 2 x SMs 128-row tiles, 8 rows for group-wise scales; 1 = never,
 *     <= 8); it takes precedence over mma_min_m.  force_threads_per_row 2,
 *     4 or 8 sets that kernel's threads per weight row (row-wise scales;
 *     the group-scale kernel always has one).
 *   mma_e4m3: operands of the row-wise tensor-core kernel: 0 = default
 *     (e4m3), 1 = binary16 (kind::f16, K = 16 per MMA), 2 = e4m3
 *     (kind::f8f6f4, K = 32 per MMA: weight bytes q + 8 read as (q + 8) *
 *     2^-9, activation codes split as 16 a_hi + a_lo).
 *   qmma_max_m: activation rows up to which row-wise W4A8 calls use the
 *     warp-level e4m3 MMA kernel, from 2 rows, on any matrix (<= 32); it
 *     takes precedence over rowdot_max_m and mma_min_m.  0 = default (2..4
 *     rows on matrices of at least 4 x SMs tiles in one K piece), 1 = never.
 *   qmma_tiles_per_warp: 16-row weight tiles per warp of that kernel (1, 2,
 *     or 4 for at most 16 rows; 0 = default).
 *   stall_test_us: for tests of the bounded waits (0 = off, <= 1 s): the
 *     warp-level MMA kernel's warps first wait, with this limit in
 *     microseconds, for a barrier phase that nothing completes.  The wait
 *     runs out, sets bit 0 of the device error word and stops the call (its
 *     outputs unspecified); copies already in flight are waited for (with
 *     the usual limit) before the kernel exits.
 *   qmma_operands: operand type of the warp-level MMA kernel: 0 = default
 *     (e4m3), 1 = binary16 (mma.sync m16n8k16: each weight code and
 *     activation code an exact binary16 integer, 8 batch rows an n-tile),
 *     2 = e4m3 (m16n8k32: weight bytes q + 8 read as (q + 8) * 2^-9,
 *     activation codes split as 16 a_hi + a_lo, 4 batch rows an n-tile).
 *     Measured on GB300: e4m3 is faster on lm_head at 2..4 rows (the
 *     default route: 57.5 vs 65.8 us at 2 rows), binary16 at 5..32 rows
 *     (gate 3584 -> 18944 at 8 rows 12.5 vs 14.8 us, lm_head at 16 rows
 *     84.5 vs 126.0), where the tensor cores lead on every matrix but gate.
 * w4a8_workspace_bytes reflects the overrides.  NULL restores the defaults.
 * Not synchronised with calls running on other threads. */
typedef struct {
    int force_splits;
    int force_threads_per_row;
    int ring_bytes;
    int ctas_per_sm;
    int mma_min_m;
    int rowdot_max_m;
    int mma_e4m3;
    int qmma_max_m;
    int qmma_tiles_per_warp;
    int stall_test_us;
    int qmma_operands;
} w4a8_tuning_t;

int w4a8_set_tuning(const w4a8_tuning_t* tuning);

/* Writes up to n_info integers describing the plan the linear entry points
 * would use for this shape, in this order: splits P, threads per row-piece,
 * granule columns per thread, row-pieces per stage, CTAs per piece, grid
 * size, most rows per CTA, ring stages, bytes per stage, dynamic shared
 * memory bytes, workspace bytes (saturated at INT32_MAX), and 1 when the
 * tensor-core kernel serves the call (then the fields read: K pieces, 0,
 * batch rows padded to 16, 128 weight rows per tile, tiles, grid, 128,
 * ring stages, bytes per stage, shared memory, workspace), or 2 when the
 * row-per-thread kernel serves it (K pieces, threads per weight row, batch
 * rows, 128, tiles, grid, 128, ring stages, 16384, shared memory,
 * workspace).  w8a16 != 0
 * selects w8a16_gemv.  num_sms > 0 plans for a device with that many SMs
 * without touching any GPU (host-side testing); 0 queries the current
 * device. */
int w4a8_plan_info(int64_t M, int64_t K, int64_t N, int w8a16, int num_sms, int* info,
                   int n_info);

/* The same for w4a8g_gemv / w4a8g_linear (the kernel field reads 1 for the
 * tensor cores, 2 for the one-thread-per-row kernel, whose threads-per-row
 * field reads 1 and whose rows field gives the batch rows of one launch),
 * followed by two more: the number of fold chunks and their length in
 * codes (max(group, 1024)). */
int w4a8g_plan_info(int64_t M, int64_t K, int64_t N, int64_t group, int num_sms, int* info,
                    int n_info);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H */

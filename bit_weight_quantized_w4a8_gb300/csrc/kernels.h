// kernels.h -- host-side launchers of the CUDA kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "qmma_plan.h"
#include "rowdot_plan.h"

namespace w4a8 {

cudaError_t launch_w4_quantize(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* sw,
                               cudaStream_t stream);
cudaError_t launch_w4g_quantize(const float* W, int64_t N, int64_t K, int gs, int64_t ld,
                                uint8_t* Wq, float* sg, cudaStream_t stream);
cudaError_t launch_w8_quantize(const float* W, int64_t N, int64_t K, int8_t* Wq8, uint16_t* sw16,
                               cudaStream_t stream);
cudaError_t launch_act_quantize(const uint16_t* X, int64_t M, int64_t K, int8_t* Xq, float* sa,
                                cudaStream_t stream);

cudaError_t launch_w4a8(const GemvPlan& pl, bool fused, const uint16_t* X, const int8_t* Xq,
                        const float* sa, int M, int64_t K, const uint8_t* Wq, const float* sw,
                        int64_t N, float* Y, int32_t* acc_out, int8_t* Xq_out, float* sa_out,
                        void* ws, unsigned flags, cudaStream_t stream, const void* pf = nullptr,
                        int64_t pf_bytes = 0);
// pf, pf_bytes: the next launch's first weight bytes to bring into L2 (see
// w4a8_linear_prefetch); pf must be 16-byte aligned.
cudaError_t launch_w4a8_grouped(const GemvPlan& pl, const uint16_t* X, int M, int64_t K, int G,
                                const uint8_t* const* Wq, const float* const* sw,
                                const int64_t* Ns, float* const* Y, void* ws, unsigned flags,
                                cudaStream_t stream, const void* pf = nullptr, int64_t pf_bytes = 0);
cudaError_t launch_w8a16(const GemvPlan& pl, const uint16_t* X, int M, int64_t K,
                         const int8_t* Wq8, const uint16_t* sw16, int64_t N, float* Y, void* ws,
                         unsigned flags, cudaStream_t stream);

cudaError_t read_and_clear_device_error(unsigned* flags, cudaStream_t stream);


// Tensor-core path (mma.cu).  make_mma_plan is host-only and needs no GPU.
// gkb > 0: group-wise scales, groups of gkb 64-code K blocks (gs = 64 gkb).
bool make_mma_plan(int M, int64_t K, int64_t N, int num_sms, MmaPlan* out, int gkb = 0, int force_p = 0);
// gs > 0: group-wise scales sg[g] ([N][stride] fp32, gs a multiple of 128,
// at most 16384); sw is then unused.
cudaError_t launch_w4a8_mma(const MmaPlan& pl, const uint16_t* X, const int8_t* Xq, const float* sa,
                            int M, int64_t K, int G, const uint8_t* const* Wq,
                            const float* const* sw, const int64_t* Ns, float* const* Y,
                            int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                            unsigned flags, cudaStream_t stream, int gs = 0,
                            const float* const* sg = nullptr, bool e4m3 = false);
cudaError_t read_and_clear_mma_error(unsigned* flags, cudaStream_t stream);
// Tensor map of packed INT4 weights [N][K/2] for 2-D TMA boxes of 128 bytes
// (256 codes) x 128 rows, 128-byte swizzle; `map` is a 64-byte aligned
// CUtensorMap.  Host-only; false when the driver entry point is missing.
bool make_w4_tile_map(void* map, const uint8_t* Wq, int64_t K, int64_t N);

// Row-per-thread dp4a kernel for small batches (rowdot.cu).
bool make_rowdot_plan(int M, int64_t K, int64_t N, int num_sms, RowdotPlan* out, int tpr = 0,
                      int cps = 0, int gshift = -1, int force_p = 0);
cudaError_t launch_w4a8_rowdot(const RowdotPlan& pl, const uint16_t* X, const int8_t* Xq,
                               const float* sa, int M, int64_t K, int G, const uint8_t* const* Wq,
                               const float* const* sw, const int64_t* Ns, float* const* Y,
                               int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                               unsigned flags, cudaStream_t stream, int gs = 0,
                               const float* const* sg = nullptr);
cudaError_t read_and_clear_rowdot_error(unsigned* flags, cudaStream_t stream);

// Warp-level e4m3 MMA kernel for small batches (qmma.cu).  make_qmma_plan
// is host-only and needs no GPU; R = 16-row tiles per warp (1, 2 or 4; 0 =
// the default for the batch size).
bool make_qmma_plan(int M, int64_t K, int64_t N, int num_sms, QmmaPlan* out, int R = 0, bool h16 = false);
cudaError_t launch_w4a8_qmma(const QmmaPlan& pl, const uint16_t* X, const int8_t* Xq, const float* sa,
                             int M, int64_t K, int G, const uint8_t* const* Wq,
                             const float* const* sw, const int64_t* Ns, float* const* Y,
                             int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                             unsigned flags, cudaStream_t stream,
                             unsigned long long stall_ns = 0);
cudaError_t read_and_clear_qmma_error(unsigned* flags, cudaStream_t stream);

// The MLP's gated product (gemv.cu, silu.cu): the one-row GEMV over an
// interleaved gate/up matrix with the product in its epilogue (a plan made
// with pair = true), and the stand-alone kernel
// h[m][i] = binary16(silu(g[m * ld + i * stride]) * u[m * ld + i * stride]).
cudaError_t launch_w4a8_silu(const GemvPlan& pl, const uint16_t* X, int M, int64_t K, const uint8_t* Wq,
                             const float* sw, int64_t N2, float* Y, uint16_t* H, void* ws, unsigned flags,
                             cudaStream_t stream);
cudaError_t launch_silu_mul(const float* g, const float* u, int64_t n, int64_t M, int64_t stride, int64_t ld,
                            uint16_t* h, unsigned flags, cudaStream_t stream);

// IndexSoftmax (isx.cu).  The host helpers need no GPU.
constexpr int kIsxMaxEntries = 256;  // 2^b table entries, b <= 8
void isx_build_lut(int b, double c, uint8_t* lut);
int64_t isx_c_int(double c, int64_t d, float s_q, float s_k);
void isx_thresholds(uint32_t c_int, int b, uint32_t* thr);
int isx_kernel_kind(int64_t cols, bool vec_ok, int* q_needed);
cudaError_t launch_index_softmax(const int32_t* A, int64_t rows, int64_t cols, uint32_t c_int,
                                 int b, const uint8_t* lut, const uint32_t* thr, uint8_t* P,
                                 cudaStream_t stream);

}  // namespace w4a8

// gemv.cu -- launchers of the streaming GEMV kernel (gemv_kernel.cuh) for
// row-wise INT4 weights (W4A8, fused and unfused) and INT8 weights (W8A16).
#include "gemv_kernel.cuh"

namespace w4a8 {

// M == 1 fused W4A8: the common column counts get kernels with exactly that
// many columns (7: K = 3584 at 16 threads per row; 5: K = 18944 at 128).
static cudaError_t launch_w4a8_m1_fused(const GemvArgs& a, unsigned flags, cudaStream_t stream) {
    if (a.pl.S == 7) return launch_one<true, 1, 7, true, true>(a, flags, stream);
    if (a.pl.S == 5) return launch_one<true, 1, 5, true, true>(a, flags, stream);
    return launch_one<true, 1, 8, true>(a, flags, stream);
}

// The prefetch hint: whole 16-byte units, shared out over the grid's CTAs.
static void set_prefetch(GemvArgs& a, const GemvPlan& pl, const void* pf, int64_t pf_bytes) {
    a.pf = static_cast<const uint8_t*>(pf);
    a.pf_bytes = pf ? pf_bytes & ~(int64_t)15 : 0;
    a.pf_share = ((a.pf_bytes + pl.grid - 1) / pl.grid + 15) & ~(int64_t)15;
}

cudaError_t launch_w4a8_grouped(const GemvPlan& pl, const uint16_t* X, int M, int64_t K, int G,
                                const uint8_t* const* Wq, const float* const* sw,
                                const int64_t* Ns, float* const* Y, void* ws, unsigned flags,
                                cudaStream_t stream, const void* pf, int64_t pf_bytes) {
    GemvArgs a = {};
    set_prefetch(a, pl, pf, pf_bytes);
    const void* s[kMaxSegments] = {};
    for (int k = 0; k < G; ++k) s[k] = sw[k];
    set_segments(a, G, Wq, s, Ns, Y);
    a.X = reinterpret_cast<const __half*>(X);
    a.tickets = static_cast<unsigned*>(ws);
    a.part = ws ? static_cast<uint8_t*>(ws) + kTicketBytes : nullptr;
    a.M = M;
    a.K = (int)K;
    a.N = (int)a.off[kMaxSegments];
    a.pl = pl;
    switch (pl.MT) {
        case 1: return launch_w4a8_m1_fused(a, flags, stream);
        case 2: return launch_one<true, 2, 4, true>(a, flags, stream);
        case 4: return launch_one<true, 4, 2, true>(a, flags, stream);
        case 8: return launch_one<true, 8, 1, true>(a, flags, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_w4a8(const GemvPlan& pl, bool fused, const uint16_t* X, const int8_t* Xq,
                        const float* sa, int M, int64_t K, const uint8_t* Wq, const float* sw,
                        int64_t N, float* Y, int32_t* acc_out, int8_t* Xq_out, float* sa_out,
                        void* ws, unsigned flags, cudaStream_t stream, const void* pf, int64_t pf_bytes) {
    GemvArgs a = {};
    set_prefetch(a, pl, pf, pf_bytes);
    const void* s0 = sw;
    set_segments(a, 1, &Wq, &s0, &N, &Y);
    a.Xq = Xq;
    a.sa = sa;
    a.X = reinterpret_cast<const __half*>(X);
    a.acc_out = acc_out;
    a.Xq_out = Xq_out;
    a.sa_out = sa_out;
    a.tickets = static_cast<unsigned*>(ws);
    a.part = ws ? static_cast<uint8_t*>(ws) + kTicketBytes : nullptr;
    a.M = M;
    a.K = (int)K;
    a.N = (int)N;
    a.pl = pl;
    switch (pl.MT * 2 + (fused ? 1 : 0)) {
        case 2: return launch_one<true, 1, 8, false>(a, flags, stream);
        case 3: return launch_w4a8_m1_fused(a, flags, stream);
        case 4: return launch_one<true, 2, 4, false>(a, flags, stream);
        case 5: return launch_one<true, 2, 4, true>(a, flags, stream);
        case 8: return launch_one<true, 4, 2, false>(a, flags, stream);
        case 9: return launch_one<true, 4, 2, true>(a, flags, stream);
        case 16: return launch_one<true, 8, 1, false>(a, flags, stream);
        case 17: return launch_one<true, 8, 1, true>(a, flags, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_w8a16(const GemvPlan& pl, const uint16_t* X, int M, int64_t K,
                         const int8_t* Wq8, const uint16_t* sw16, int64_t N, float* Y, void* ws,
                         unsigned flags, cudaStream_t stream) {
    GemvArgs a = {};
    const uint8_t* w0 = reinterpret_cast<const uint8_t*>(Wq8);
    const void* s0 = sw16;
    set_segments(a, 1, &w0, &s0, &N, &Y);
    a.X = reinterpret_cast<const __half*>(X);
    a.tickets = static_cast<unsigned*>(ws);
    a.part = ws ? static_cast<uint8_t*>(ws) + kTicketBytes : nullptr;
    a.M = M;
    a.K = (int)K;
    a.N = (int)N;
    a.pl = pl;
    switch (pl.MT) {
        case 1:  // exact column counts for K = 4096 (8 at 32 threads per row) and 13696 (7 at 128)
            if (pl.S == 8) return launch_one<false, 1, 8, false, true>(a, flags, stream);
            if (pl.S == 7) return launch_one<false, 1, 7, false, true>(a, flags, stream);
            return launch_one<false, 1, 8, false>(a, flags, stream);
        case 2: return launch_one<false, 2, 4, false>(a, flags, stream);
        case 4: return launch_one<false, 4, 2, false>(a, flags, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_and_clear_device_error(unsigned* flags, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(flags, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
}

}  // namespace w4a8

namespace w4a8 {

// One-row fused W4A8 linear on an interleaved gate/up matrix (rows 2i =
// gate i, 2i + 1 = up i, N2 rows) whose epilogue also writes the gated
// products H[m][i] = binary16(silu(Y[m][2i]) * Y[m][2i+1]).  The plan must
// have been made with pair = true.
cudaError_t launch_w4a8_silu(const GemvPlan& pl, const uint16_t* X, int M, int64_t K, const uint8_t* Wq,
                             const float* sw, int64_t N2, float* Y, uint16_t* H, void* ws, unsigned flags,
                             cudaStream_t stream) {
    GemvArgs a = {};
    const void* s0 = sw;
    set_segments(a, 1, &Wq, &s0, &N2, &Y);
    a.X = reinterpret_cast<const __half*>(X);
    a.H = reinterpret_cast<__half*>(H);
    a.tickets = static_cast<unsigned*>(ws);
    a.part = ws ? static_cast<uint8_t*>(ws) + kTicketBytes : nullptr;
    a.M = M;
    a.K = (int)K;
    a.N = (int)N2;
    a.pl = pl;
    switch (pl.MT) {
        case 1: return launch_w4a8_m1_fused(a, flags, stream);
        case 2: return launch_one<true, 2, 4, true>(a, flags, stream);
        case 4: return launch_one<true, 4, 2, true>(a, flags, stream);
        case 8: return launch_one<true, 8, 1, true>(a, flags, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4a8

// gemv_group.cu -- launchers of the streaming GEMV kernel (gemv_kernel.cuh)
// for INT4 weights with group-wise scales (the Jetson INT4 page, section
// 后续优化方向): one fp32 scale per group of gs codes along K, gs a power of
// two from 32, scale rows padded to a multiple of 4 floats.
#include "gemv_kernel.cuh"

namespace w4a8 {

// M == 1 fused: exact column counts for K = 3584 (7) and K = 18944 (5).
static cudaError_t launch_group_m1_fused(const GemvArgs& a, unsigned flags, cudaStream_t stream) {
    if (a.pl.S == 7) return launch_one<true, 1, 7, true, true, true>(a, flags, stream);
    if (a.pl.S == 5) return launch_one<true, 1, 5, true, true, true>(a, flags, stream);
    return launch_one<true, 1, 8, true, false, true>(a, flags, stream);
}

cudaError_t launch_w4a8g(const GemvPlan& pl, bool fused, const uint16_t* X, const int8_t* Xq,
                         const float* sa, int M, int64_t K, int gs, int G,
                         const uint8_t* const* Wq, const float* const* sg, const int64_t* Ns,
                         float* const* Y, int8_t* Xq_out, float* sa_out, void* ws,
                         unsigned flags, cudaStream_t stream) {
    if (G < 1 || G > kMaxSegments || gs < 32 || (gs & (gs - 1)) || K % gs)
        return cudaErrorInvalidValue;
    GemvArgs a = {};
    const void* s[kMaxSegments] = {};
    for (int k = 0; k < G; ++k) s[k] = sg[k];
    set_segments(a, G, Wq, s, Ns, Y);
    a.X = reinterpret_cast<const __half*>(X);
    a.Xq = Xq;
    a.sa = sa;
    a.Xq_out = Xq_out;
    a.sa_out = sa_out;
    a.tickets = static_cast<unsigned*>(ws);
    a.part = ws ? static_cast<uint8_t*>(ws) + kTicketBytes : nullptr;
    a.M = M;
    a.K = (int)K;
    a.N = (int)a.off[kMaxSegments];
    int gshift = 0;
    while ((32 << gshift) < gs) ++gshift;
    a.gshift = gshift;
    a.gld = (int)((K / gs + 3) / 4 * 4);
    a.pl = pl;
    switch (pl.MT * 2 + (fused ? 1 : 0)) {
        case 2: return launch_one<true, 1, 8, false, false, true>(a, flags, stream);
        case 3: return launch_group_m1_fused(a, flags, stream);
        case 4: return launch_one<true, 2, 4, false, false, true>(a, flags, stream);
        case 5: return launch_one<true, 2, 4, true, false, true>(a, flags, stream);
        case 8: return launch_one<true, 4, 2, false, false, true>(a, flags, stream);
        case 9: return launch_one<true, 4, 2, true, false, true>(a, flags, stream);
        case 16: return launch_one<true, 8, 1, false, false, true>(a, flags, stream);
        case 17: return launch_one<true, 8, 1, true, false, true>(a, flags, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_and_clear_group_error(unsigned* flags, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    *flags |= v;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
}

}  // namespace w4a8

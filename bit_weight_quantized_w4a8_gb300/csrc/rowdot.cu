// rowdot.cu -- W4A8 linear for small decode batches (2..8 activation rows)
// on the integer pipe, one weight row per thread group.
//
// The arithmetic is the W4A8 contract of the Jetson INT4 page (sections
// 正确方向 / 当前实现方式): INT8 activation codes times INT4 weight codes,
// summed exactly in int32, y = ((float)acc * s_w) * s_a.
//
// Where the dp4a GEMV spreads one weight row over a warp (each lane its own
// K slice, its own activation values), this kernel gives each weight row to
// TPR threads of one warp and walks the whole K piece with them: every
// thread of the CTA then reads the same activation words at the same time
// (shared-memory broadcasts), so the activations cost one load per batch
// row per 16 bytes for the whole warp, and the weight codes are unpacked
// once for all batch rows.  Per packed word w (8 INT4 codes, two's
// complement nibbles, low nibble first):
//   lo = (w << 4) & 0xF0F0F0F0   -> bytes 16 * q of the even codes
//   hi =  w       & 0xF0F0F0F0   -> bytes 16 * q of the odd codes
// both signed bytes, so two signed dp4a against the even and odd
// activation codes add 16 * (the 8 products) to the accumulator with no
// correction term; the sum is a multiple of 16 and >> 4 recovers it.
// |16 q a| <= 16256, so a thread's sum over at most 131072 codes stays
// inside int32.
//
// Two kernels:
//  * rowdot_codes_kernel (grid: batch rows x pieces of 2048 codes): the
//    per-row INT8 quantization of the activations (max|x|, s_a = max/127 by
//    IEEE division, round half away, clamp; actq.cuh), or the given int8
//    codes, written split by parity: per 8 codes one 8-byte word pair (the
//    4 even codes, the 4 odd codes), zero past K up to a whole 256-code box,
//    and interleaved over the batch: the 32 codes of one 16-byte weight
//    chunk are 32 contiguous bytes per batch row, the M rows of a chunk
//    adjacent ([box][chunk][M][32 bytes]).
//  * rowdot_kernel<MT, TPR> (one CTA per 128 weight rows and K piece):
//    thread 0 streams 2-D TMA boxes of 128 rows x 128 bytes (256 codes,
//    128-byte swizzle) into a ring and copies the piece's activation planes
//    once; each thread group accumulates its row's dot products with all
//    MT batch rows; pieces are summed in int32 by the CTA that finishes a
//    tile last (exact, so the result is bit-identical to the integer
//    definition whatever the split).  With group-wise scales (kG) every
//    32-code granule's exact sum is folded into an fp32 sum with its group
//    scale (staged per CTA), and the sums are added in a fixed order.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>

#include "actq.cuh"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace w4a8 {

__device__ unsigned g_rowdot_error;  // wait timeouts of this path (same bits as the GEMV's)

namespace {

constexpr int kTile = 128;             // weight rows per CTA
constexpr int kBoxCodes = 256;         // K codes per TMA box (128 bytes of a row)
constexpr int kBoxBytes = kTile * kBoxCodes / 2;  // 16384
constexpr int kActBoxBytes = kBoxCodes;           // activation bytes of one batch row per box
constexpr int kPreThreads = 256;
constexpr int kMaxNS = 8;
constexpr int kActMax = 48 * 1024;     // shared bytes for a piece's activation codes
constexpr int kSmemPerSM = 227 * 1024;

struct RowdotArgs {
    CUtensorMap tmW;        // packed weights [N][K/2] uint8, box 128 bytes x 128 rows, 128B swizzle
    const uint2* codes;     // activation codes [nbox][8][M][4] (even, odd) word pairs
    const float* sw;        // [N]
    const float* sa;        // [M]
    float* Y;               // [M][N]
    int32_t* acc_out;       // optional [M][N]
    int32_t* part;          // [tiles][P][M][128] piece sums when P > 1 (int32; fp32 with group scales)
    unsigned* tickets;      // [tiles] when P > 1, zero between calls
    // group scales: sg [N][gld] fp32, one per 2^gshift codes, ngroups = K >> gshift;
    // a piece's window of gwin groups is staged per CTA as [128][gstride]
    const float* sg;
    int gshift, gld, ngroups, gwin, gstride;
    int M, N, nbox, bpp, P, NS;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        #pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(&g_rowdot_error, kErrFullWait);
            return false;
        }
    }
}

// Activation codes.  Grid (M rows, ceil(kw / 256)); thread u handles the
// 8 codes 8u..8u+7 of row m.  Every CTA of a row takes the row's max|x|
// (exact in binary16) and s_a = max/127 by IEEE division, then quantizes its
// vectors with the fast exact quantizer; with X null it splits the given
// int8 codes Xq instead.  Optional int8 codes and scale outputs.
__global__ void __launch_bounds__(kPreThreads) rowdot_codes_kernel(
    const __half* __restrict__ X, const int8_t* __restrict__ Xq, const float* __restrict__ sa_in,
    int M, int64_t K, int64_t kw, uint2* __restrict__ codes, float* __restrict__ sa_ws,
    int8_t* __restrict__ Xq_out, float* __restrict__ sa_out) {
    __shared__ float red[kPreThreads / 32];
    griddep_launch_dependents();
    griddep_wait();
    const int m = blockIdx.x;
    const int64_t u = (int64_t)blockIdx.y * kPreThreads + threadIdx.x;
    const int64_t kchunks = K / 8;
    float s;
    const uint4* xv = reinterpret_cast<const uint4*>(X + (int64_t)m * K);
    if (X == nullptr) {
        s = sa_in[m];
    } else {
        __half2 hm = __float2half2_rn(0.f);
        #pragma unroll 4
        for (int64_t v = threadIdx.x; v < kchunks; v += kPreThreads) {
            const uint4 h = xv[v];
            const __half2* p2 = reinterpret_cast<const __half2*>(&h);
            #pragma unroll
            for (int t = 0; t < 4; ++t) hm = __hmax2(hm, __habs2(p2[t]));
        }
        float mx = fmaxf(__low2float(hm), __high2float(hm));
        #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = 0.f;
        #pragma unroll
        for (int w = 0; w < kPreThreads / 32; ++w) mx = fmaxf(mx, red[w]);
        s = __fdiv_rn(mx, 127.f);
    }
    if (u < kw) {
        uint2 q = make_uint2(0u, 0u);
        if (u < kchunks) {
            if (X != nullptr) {
                float r_lo, r_hi;
                quant_bracket(s, &r_lo, &r_hi);
                q = quant8_split(xv[u], s, r_lo, r_hi);  // even / odd codes
                if (Xq_out != nullptr)
                    *reinterpret_cast<uint2*>(Xq_out + (int64_t)m * K + 8 * u) =
                        make_uint2(__byte_perm(q.x, q.y, 0x5140), __byte_perm(q.x, q.y, 0x7362));
            } else {
                const uint2 c = *reinterpret_cast<const uint2*>(Xq + (int64_t)m * K + 8 * u);
                q = make_uint2(__byte_perm(c.x, c.y, 0x6420), __byte_perm(c.x, c.y, 0x7531));
            }
        }
        // word pair u = (box, chunk, j): [box][chunk][m][j]
        codes[((u >> 2) * M + m) * 4 + (u & 3)] = q;
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) {
        sa_ws[m] = s;
        if (sa_out != nullptr) sa_out[m] = s;
    }
}

// Shared memory (base aligned to 1024 for the swizzled boxes): the weight
// ring [NS][16384], the piece's activation codes [bpp][8][MT][32 bytes], the
// cross-warp sums [TPR - 1][MT][128] (int32; fp32 with group scales), with
// group scales the piece's scale window [128][gstride] fp32, NS + 1 mbarriers
// (ring slots, activations), and per slot the number of warps done with it
// and the last box copied into it.
//
// Thread mapping: warp w takes the 16-byte chunks c = w / 4 + TPR * i of
// every 128-byte box row, lane l the weight row r = (w % 4) * 32 + l.  With
// the 128-byte swizzle (chunk c of row r stored at r * 128 + ((c ^ (r % 8))
// * 16)) the eight lanes of each quarter-warp read eight different bank
// groups (conflict-free), and every activation load of a warp is one
// address (a broadcast).
//
// kG (group-wise scales, groups of 2^gshift >= 32 codes): a 32-code chunk is
// one granule of one group; its exact int32 sum v is folded into an fp32 sum
// per batch row with one fma(v, s_g, sum), the four threads of a row add
// their fp32 sums in a fixed order, pieces add theirs in piece order, and
// the result is multiplied by s_a.
template <int MT, int TPR, bool kG>
__global__ void __launch_bounds__(kTile * TPR) rowdot_kernel(const __grid_constant__ RowdotArgs a) {
    constexpr int kThreads = kTile * TPR;
    constexpr int kWarps = kThreads / 32;
    constexpr int CPT = 8 / TPR;           // chunks of each box row per thread
    constexpr int kChunkAct = MT * 32;     // activation bytes of one chunk
    constexpr int kBoxAct = 8 * kChunkAct; // activation bytes of one box
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int NS = a.NS;
    uint8_t* ring = smem;
    uint8_t* act = smem + NS * kBoxBytes;
    int* red = reinterpret_cast<int*>(act + a.bpp * kBoxAct);
    float* sgs = reinterpret_cast<float*>(red + (TPR - 1) * MT * kTile);  // group scales
    uint64_t* bars = reinterpret_cast<uint64_t*>(sgs + (kG ? kTile * a.gstride : 0));  // full[NS], activations
    int* released = reinterpret_cast<int*>(bars + NS + 1);
    int* last_box = released + NS;
    volatile int* abort_flag = last_box + NS;
    int* last_flag = last_box + NS + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / a.P, p = blockIdx.x % a.P;
    const int box0 = p * a.bpp;
    const int nb = min(a.bpp, a.nbox - box0);
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint64_t pol = l2_evict_first_policy();
    const int g0 = kG ? (box0 * kBoxCodes) >> a.gshift : 0;  // first group of the piece

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(bars + s), 1);
            released[s] = 0;
            last_box[s] = -1;
        }
        mbar_init(smem_u32(bars + NS), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    if (tid == 0) {  // the weights do not depend on earlier launches
        const int n0 = min(NS, nb);
        for (int i = 0; i < n0; ++i) {
            mbar_arrive_expect_tx(smem_u32(bars + i), kBoxBytes);
            tma_load_2d_hint(smem_u32(ring + i * kBoxBytes), &a.tmW, (box0 + i) * (kBoxCodes / 2),
                             tile * kTile, smem_u32(bars + i), pol);
            last_box[i] = i;
        }
    }
    if constexpr (kG) {
        // the piece's scale window; zero for rows past N and groups past K
        for (int e = tid; e < kTile * a.gwin; e += kThreads) {
            const int rr = e / a.gwin, j = e - rr * a.gwin;
            const int64_t n = (int64_t)tile * kTile + rr;
            float* dst = sgs + rr * a.gstride + j;
            if (n < a.N && g0 + j < a.ngroups)
                cp_async_4(smem_u32(dst), a.sg + n * a.gld + g0 + j);
            else
                *dst = 0.f;
        }
    }
    griddep_wait();  // activation codes, scales, outputs and workspace from here on
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)nb * kBoxAct;
        mbar_arrive_expect_tx(smem_u32(bars + NS), bytes);
        bulk_g2s(smem_u32(act), reinterpret_cast<const uint8_t*>(a.codes) + (int64_t)box0 * kBoxAct, bytes,
                 smem_u32(bars + NS), l2_evict_last_policy());
    }
    if constexpr (kG) {
        cp_async_wait_all();
        __syncthreads();
    }

    int acc[MT][2];  // 16 x the even / odd products of each batch row
    float gacc[kG ? MT : 1];  // group scales: fp32 sums of scaled granules
    #pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0;
    #pragma unroll
    for (int m = 0; m < (kG ? MT : 1); ++m) gacc[m] = 0.f;
    const uint8_t* wrow = ring + r * 128;
    bool ok = wait_bounded(smem_u32(bars + NS), 0, abort_flag);
    int slot = 0;
    uint32_t ph = 0;
    for (int i = 0; ok && i < nb; ++i) {
        if (!wait_bounded(smem_u32(bars + slot), ph, abort_flag)) break;
        uint4 wv[CPT];
        #pragma unroll
        for (int ci = 0; ci < CPT; ++ci) {
            const int c = t + TPR * ci;
            wv[ci] = *reinterpret_cast<const uint4*>(wrow + slot * kBoxBytes + ((c ^ (r & 7)) << 4));
        }
        __syncwarp();
        if (lane == 0) {
            // the last warp done with this slot refills it with the box NS further on
            __threadfence_block();
            if (atomicAdd(released + slot, 1) == kWarps - 1) {
                released[slot] = 0;
                __threadfence_block();
                if (i + NS < nb && !*abort_flag) {
                    mbar_arrive_expect_tx(smem_u32(bars + slot), kBoxBytes);
                    tma_load_2d_hint(smem_u32(ring + slot * kBoxBytes), &a.tmW,
                                     (box0 + i + NS) * (kBoxCodes / 2), tile * kTile, smem_u32(bars + slot), pol);
                    last_box[slot] = i + NS;
                }
            }
        }
        if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
        }
        const uint8_t* ab = act + i * kBoxAct;
        #pragma unroll
        for (int ci = 0; ci < CPT; ++ci) {
            const int c = t + TPR * ci;
            const uint8_t* ac = ab + c * kChunkAct;
            const uint32_t w[4] = {wv[ci].x, wv[ci].y, wv[ci].z, wv[ci].w};
            int lo[4], hi[4];
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo[j] = (int)((w[j] << 4) & 0xF0F0F0F0u);
                hi[j] = (int)(w[j] & 0xF0F0F0F0u);
            }
            if constexpr (kG) {
                #pragma unroll
                for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0;
            }
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 a0 = *reinterpret_cast<const uint4*>(ac + m * 32);
                const uint4 a1 = *reinterpret_cast<const uint4*>(ac + m * 32 + 16);
                acc[m][0] = __dp4a(lo[0], (int)a0.x, acc[m][0]);
                acc[m][1] = __dp4a(hi[0], (int)a0.y, acc[m][1]);
                acc[m][0] = __dp4a(lo[1], (int)a0.z, acc[m][0]);
                acc[m][1] = __dp4a(hi[1], (int)a0.w, acc[m][1]);
                acc[m][0] = __dp4a(lo[2], (int)a1.x, acc[m][0]);
                acc[m][1] = __dp4a(hi[2], (int)a1.y, acc[m][1]);
                acc[m][0] = __dp4a(lo[3], (int)a1.z, acc[m][0]);
                acc[m][1] = __dp4a(hi[3], (int)a1.w, acc[m][1]);
            }
            if constexpr (kG) {
                // the granule's group scale; |v| <= 1016 * 32 is exact in fp32
                const int g = (((box0 + i) * kBoxCodes + c * 32) >> a.gshift) - g0;
                const float sgv = sgs[r * a.gstride + g];
                #pragma unroll
                for (int m = 0; m < MT; ++m)
                    gacc[m] = __fmaf_rn(__int2float_rn((acc[m][0] >> 4) + (acc[m][1] >> 4)), sgv, gacc[m]);
            }
        }
    }

    // The row's sums: integers (the two dp4a sums are 16 x integers), or fp32
    // with group scales; the warps of chunk phases t > 0 hand theirs to
    // phase 0, which adds them in phase order.
    int v[MT];
    if constexpr (kG) {
        #pragma unroll
        for (int m = 0; m < MT; ++m) v[m] = __float_as_int(gacc[m]);
    } else {
        #pragma unroll
        for (int m = 0; m < MT; ++m) v[m] = (acc[m][0] >> 4) + (acc[m][1] >> 4);
    }
    if (t > 0) {
        #pragma unroll
        for (int m = 0; m < MT; ++m) red[((t - 1) * MT + m) * kTile + r] = v[m];
    }
    __syncthreads();
    if (*abort_flag && tid == 0) {
        // copies may still be landing after an abandoned wait: wait for the
        // last one of each slot (bounded) so none writes shared memory after exit
        if (!mbar_wait(smem_u32(bars + NS), 0)) atomicOr(&g_rowdot_error, kErrDrainWait);
        for (int s = 0; s < NS; ++s)
            if (last_box[s] >= 0 && !mbar_wait(smem_u32(bars + s), (uint32_t)(last_box[s] / NS) & 1u))
                atomicOr(&g_rowdot_error, kErrDrainWait);
    }
    if (t == 0) {
        #pragma unroll
        for (int tt = 1; tt < TPR; ++tt) {
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                const int o = red[((tt - 1) * MT + m) * kTile + r];
                if constexpr (kG)
                    v[m] = __float_as_int(__fadd_rn(__int_as_float(v[m]), __int_as_float(o)));
                else
                    v[m] += o;
            }
        }
    }
    const int n = tile * kTile + r;
    if (a.P == 1) {
        if (t == 0 && n < a.N) {
            const float swv = kG ? 0.f : a.sw[n];
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                if constexpr (kG) {
                    a.Y[(int64_t)m * a.N + n] = __fmul_rn(__int_as_float(v[m]), a.sa[m]);
                } else {
                    a.Y[(int64_t)m * a.N + n] = __fmul_rn(__fmul_rn(__int2float_rn(v[m]), swv), a.sa[m]);
                    if (a.acc_out != nullptr) a.acc_out[(int64_t)m * a.N + n] = v[m];
                }
            }
        }
        return;
    }

    // ------------------------------------------------ split K: last CTA sums
    if (t == 0) {
        int32_t* dst = a.part + ((int64_t)(tile * a.P + p) * MT) * kTile + r;
        #pragma unroll
        for (int m = 0; m < MT; ++m) dst[m * kTile] = v[m];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) *last_flag = (atomicAdd(a.tickets + tile, 1u) == (unsigned)(a.P - 1));
    __syncthreads();
    if (!*last_flag) return;
    __threadfence();
    const int32_t* src = a.part + (int64_t)tile * a.P * MT * kTile;
    for (int e = tid; e < MT * kTile; e += kThreads) {
        const int m = e / kTile, rr = e % kTile, nn = tile * kTile + rr;
        if (nn >= a.N) continue;
        if constexpr (kG) {
            float sum = 0.f;
            for (int q = 0; q < a.P; ++q)
                sum = __fadd_rn(sum, __int_as_float(__ldcg(src + (int64_t)q * MT * kTile + e)));
            a.Y[(int64_t)m * a.N + nn] = __fmul_rn(sum, a.sa[m]);
        } else {
            int32_t sum = 0;
            for (int q = 0; q < a.P; ++q) sum += __ldcg(src + (int64_t)q * MT * kTile + e);
            a.Y[(int64_t)m * a.N + nn] = __fmul_rn(__fmul_rn(__int2float_rn(sum), a.sw[nn]), a.sa[m]);
            if (a.acc_out != nullptr) a.acc_out[(int64_t)m * a.N + nn] = sum;
        }
    }
    if (tid == 0) a.tickets[tile] = 0u;  // ready for the next call
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned flags, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (flags & 1u) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int MT, int TPR, bool kG>
const void* kernel_for() {
    return reinterpret_cast<const void*>(rowdot_kernel<MT, TPR, kG>);
}

template <int TPR, bool kG>
const void* kernel_for_rows(int M) {
    switch (M) {
        case 2: return kernel_for<2, TPR, kG>();
        case 3: return kernel_for<3, TPR, kG>();
        case 4: return kernel_for<4, TPR, kG>();
        case 5: return kernel_for<5, TPR, kG>();
        case 6: return kernel_for<6, TPR, kG>();
        case 7: return kernel_for<7, TPR, kG>();
        case 8: return kernel_for<8, TPR, kG>();
        default: return nullptr;
    }
}

// Row-wise scales: 2, 4 or 8 threads per row; group scales: 4.
const void* kernel_for(int M, int tpr, bool group) {
    if (group) return tpr == 4 ? kernel_for_rows<4, true>(M) : nullptr;
    switch (tpr) {
        case 2: return kernel_for_rows<2, false>(M);
        case 4: return kernel_for_rows<4, false>(M);
        case 8: return kernel_for_rows<8, false>(M);
        default: return nullptr;
    }
}

// Opts every instantiation into its largest shared-memory plan (and the
// full shared-memory carveout, so that the planned CTAs per SM fit), once
// per device.
cudaError_t set_attributes() {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && done[dev]) return cudaSuccess;
    for (int k = 0; k < 4; ++k) {
        for (int M = 2; M <= kRowdotMaxM; ++M) {
            const void* fn = k < 3 ? kernel_for(M, 2 << k, false) : kernel_for(M, 4, true);
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPerSM - 1024);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
    }
    if (dev < 64) done[dev] = true;
    return cudaSuccess;
}

size_t smem_bytes(int M, int NS, int bpp, int tpr, int gstride) {
    return 1024 + (size_t)NS * kBoxBytes + (size_t)M * bpp * kActBoxBytes +
           (size_t)(tpr - 1) * M * kTile * 4 + (size_t)kTile * gstride * 4 + (size_t)(NS + 1) * 8 +
           (size_t)(2 * NS + 2) * 4;
}

}  // namespace

// Plan: one CTA per 128 weight rows and K piece, TPR threads per row and
// cps CTAs per SM (0 = the defaults: 4 threads, 4 / TPR CTAs).  K is split
// into pieces of whole 256-code boxes when the tiles alone leave CTA slots
// idle, and so that a piece's activation codes fit in kActMax bytes.  The
// ring takes what shared memory is left, up to kMaxNS boxes.  gshift >= 0:
// group scales (groups of 2^gshift codes, 4 threads per row), the piece's
// scale window staged per CTA.
bool make_rowdot_plan(int M, int64_t K, int64_t N, int num_sms, RowdotPlan* out, int tpr, int cps,
                      int gshift) {
    if (M < 2 || M > kRowdotMaxM || K < 32 || K % 32 || K > 131072 || N < 1 || N > 0x7FFFFFFF)
        return false;
    if (tpr == 0 || gshift >= 0) tpr = kRowdotDefaultTPR;
    if (tpr != 2 && tpr != 4 && tpr != 8) return false;
    if (gshift >= 0 && (gshift < 5 || gshift > 17 || K % (1LL << gshift))) return false;
    if (cps == 0) cps = tpr < 4 ? 4 / tpr : 1;
    if (cps < 1 || cps > 4) return false;
    RowdotPlan pl = {};
    pl.tpr = tpr;
    pl.MT = M;
    pl.tiles = (int)((N + kTile - 1) / kTile);
    pl.nbox = (int)((K + kBoxCodes - 1) / kBoxCodes);
    pl.cps = cps;
    const int slots = pl.cps * num_sms;
    int P = 1;
    if (pl.tiles < slots * 4 / 5) P = slots / pl.tiles;
    const int bpp_max = kActMax / (M * kActBoxBytes);
    const int pmin = (pl.nbox + bpp_max - 1) / bpp_max;
    if (P < pmin) P = pmin;
    if (P > pl.nbox) P = pl.nbox;
    pl.bpp = (pl.nbox + P - 1) / P;
    pl.P = (pl.nbox + pl.bpp - 1) / pl.bpp;
    if (pl.P > 1 && pl.tiles > kTicketSlots) return false;
    if ((int64_t)pl.tiles * pl.P > 0x7FFFFFFF) return false;
    pl.gshift = gshift;
    if (gshift >= 0) {
        // groups a piece touches: whole groups when boxes hold whole groups,
        // else the piece may start and end inside one
        pl.gwin = (int)(((int64_t)pl.bpp * kBoxCodes) >> gshift) + 2;
        pl.gstride = pl.gwin | 1;  // odd: the 32 rows of a warp hit 32 banks
    }
    const int budget = kSmemPerSM / pl.cps - 1024;
    int NS = kMaxNS < pl.bpp ? kMaxNS : pl.bpp;
    while (NS > 1 && smem_bytes(M, NS, pl.bpp, tpr, pl.gstride) > (size_t)budget) --NS;
    if (smem_bytes(M, NS, pl.bpp, tpr, pl.gstride) > (size_t)budget) return false;
    pl.NS = NS;
    pl.smem = (int)smem_bytes(M, NS, pl.bpp, tpr, pl.gstride);
    pl.grid = pl.tiles * pl.P;
    pl.sms = num_sms;
    // workspace: tickets, scales, activation codes [nbox][8][M][32 bytes],
    // then piece sums [tiles][P][M][128] (int32, or fp32 with group scales).
    // Sized for any N' <= N (grouped launches plan each matrix on its own):
    // a matrix is split either because its tiles leave CTA slots idle
    // (then tiles' * P' <= slots) or because a piece's codes must fit in
    // kActMax (P' = pmin, tiles' <= tiles), so max(slots, tiles * pmin)
    // tile pieces when pmin > 1, else slots.
    pl.off_sa = kTicketBytes;
    pl.off_codes = pl.off_sa + 256;
    pl.off_part = round_up_sz(pl.off_codes + (size_t)M * pl.nbox * kActBoxBytes, 256);
    int64_t units = slots;
    if (pmin > 1 && units < (int64_t)pl.tiles * pmin) units = (int64_t)pl.tiles * pmin;
    if (pl.P > 1 && units < (int64_t)pl.tiles * pl.P) units = (int64_t)pl.tiles * pl.P;
    pl.ws_bytes = pl.off_part + round_up_sz((size_t)units * M * kTile * 4, 256);
    *out = pl;
    return true;
}

cudaError_t launch_w4a8_rowdot(const RowdotPlan& pl, const uint16_t* X, const int8_t* Xq,
                               const float* sa, int M, int64_t K, int G, const uint8_t* const* Wq,
                               const float* const* sw, const int64_t* Ns, float* const* Y,
                               int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                               unsigned flags, cudaStream_t stream, int gs, const float* const* sg) {
    const bool group = gs > 0;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    float* sa_ws = reinterpret_cast<float*>(wsb + pl.off_sa);
    uint2* codes = reinterpret_cast<uint2*>(wsb + pl.off_codes);
    const int64_t kw = (int64_t)pl.nbox * (kBoxCodes / 8);
    {
        const __half* xh = reinterpret_cast<const __half*>(X);
        int Mi = M;
        int64_t Kk = K, kwv = kw;
        void* args[] = {&xh, &Xq, &sa, &Mi, &Kk, &kwv, &codes, &sa_ws, &Xq_out, &sa_out};
        const unsigned pieces = (unsigned)((kw + kPreThreads - 1) / kPreThreads);
        cudaError_t e = launch_pdl(reinterpret_cast<const void*>(rowdot_codes_kernel), dim3(M, pieces),
                                   dim3(kPreThreads), 0, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    const void* fn = kernel_for(M, pl.tpr, group);
    if (fn == nullptr || group != (pl.gshift >= 0)) return cudaErrorInvalidValue;
    cudaError_t e = set_attributes();
    if (e != cudaSuccess) return e;
    for (int g = 0; g < G; ++g) {
        RowdotPlan pg;
        if (!make_rowdot_plan(M, K, Ns[g], pl.sms, &pg, pl.tpr, pl.cps, pl.gshift)) return cudaErrorInvalidValue;
        RowdotArgs a;
        memset(&a, 0, sizeof(a));
        if (!make_w4_tile_map(&a.tmW, Wq[g], K, Ns[g])) return cudaErrorInvalidValue;
        a.codes = codes;
        a.sw = group ? nullptr : sw[g];
        if (group) {
            a.sg = sg[g];
            a.gshift = pg.gshift;
            a.gld = (int)((K / gs + 3) / 4 * 4);
            a.ngroups = (int)(K >> pg.gshift);
            a.gwin = pg.gwin;
            a.gstride = pg.gstride;
        }
        a.sa = sa_ws;
        a.Y = Y[g];
        a.acc_out = (G == 1) ? acc_out : nullptr;
        a.part = reinterpret_cast<int32_t*>(wsb + pg.off_part);
        a.tickets = reinterpret_cast<unsigned*>(wsb);
        a.M = M;
        a.N = (int)Ns[g];
        a.nbox = pg.nbox;
        a.bpp = pg.bpp;
        a.P = pg.P;
        a.NS = pg.NS;
        void* args[] = {&a};
        e = launch_pdl(fn, dim3(pg.grid), dim3(kTile * pg.tpr), pg.smem, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_and_clear_rowdot_error(unsigned* flags, cudaStream_t stream) {
    unsigned v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_rowdot_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_rowdot_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    *flags |= v;
    return e;
}

}  // namespace w4a8

// abi.cu -- the extern "C" entry points declared in include/w4a8.h:
// argument checks on the host, plan selection, launches on the caller's
// stream.  Nothing here allocates or synchronises (except
// w4a8_device_error, which is documented to synchronise).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <string>

#include "../../include/w4a8.h"
#include "kernels.h"
#include "plan.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int ok() {
    g_last_error.clear();
    return W4A8_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(W4A8_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Process-wide tuning knobs (w4a8_set_tuning); read at plan time.
std::atomic<int> g_force_splits{0};
std::atomic<int> g_force_cl{0};
std::atomic<int> g_ring_bytes{0};
std::atomic<int> g_ctas_per_sm{0};
std::atomic<int> g_mma_min_m{0};
std::atomic<int> g_rowdot_max_m{0};
std::atomic<int> g_mma_e4m3{0};
std::atomic<int> g_qmma_max_m{0};
std::atomic<int> g_qmma_r{0};
std::atomic<int> g_stall_test_us{0};
std::atomic<int> g_qmma_ops{0};  // 0 default (e4m3), 1 binary16, 2 e4m3
// Test of the bounded waits (w4a8_tuning_t.stall_test_us): 0 = off.
unsigned long long qmma_stall_ns() { return (unsigned long long)g_stall_test_us.load() * 1000ull; }
// Row-wise tensor-core calls use e4m3 operands by default: weight bytes
// q + 8 (exactly (q + 8) * 2^-9, three instructions per 8 codes) and K = 32
// per MMA, half the MMAs and TMEM stores of the binary16 path.  Measured on
// GB300 (graphs of ten calls): lm_head at 8 rows 59.7 vs 88.2 us, gate at
// 16 rows 15.9 vs 19.7 us, down at 8 rows 14.8 vs 18.8 us.
constexpr bool kDefaultMmaE4m3 = true;
bool mma_e4m3() {
    const int v = g_mma_e4m3.load();
    return v == 0 ? kDefaultMmaE4m3 : v == 2;
}
// Batch rows up to which row-wise W4A8 calls take the row-per-thread dp4a
// kernel (from 2 rows) by default, on matrices of at most two tiles per SM:
// measured on GB300 at 2 rows, gate 8.8 vs 12.6 us and down 11.9 vs 13.7 us
// on the tensor cores, but lm_head (1188 tiles) 62.3 vs 57.9 us.
constexpr int kDefaultRowdotMaxM = 3;
// Batch rows from which the W4A8 entry points take the tensor-core kernel
// when the row-per-thread kernel does not serve the call: row-wise scales
// from 2 rows (e4m3 operands), group-wise scales from 3 (binary16 operands;
// by default the one-thread-per-row kernel serves group-wise calls of 1..8
// rows, so the tensor cores take them from 9).
constexpr int kDefaultMmaMinM = 2;
constexpr int kDefaultMmaMinMGroup = 3;
// Group-wise scales: the one-thread-per-row kernel serves 1..8 rows by
// default (the tensor cores' per-group readouts make them slower there).
constexpr int kDefaultRowdotMaxMGroup = 8;
// The warp-level e4m3 MMA kernel serves row-wise W4A8 calls of 2..4 rows
// whose plan is persistent (one K piece) with at least kQmmaMinTilesPerSm
// tiles per SM: lm_head-sized matrices, where two persistent CTAs per SM
// beat the e4m3 tensor cores (GB300, graphs of ten calls, two weight
// copies: lm_head 3584 -> 152064 at 2 / 4 rows 57.3 / 59.6 vs 60.1 / 60.4
// us; at 8 rows 75.0 vs 61.6, at gate's 148 tiles slower).
// w4a8_tuning_t.qmma_max_m = 1 switches it off, >= 2 gives it every call of
// 2 rows up to that (any matrix), ahead of the two kernels above.
constexpr int kDefaultQmmaMaxM = 4;
constexpr int kQmmaMinTilesPerSm = 4;

int sm_count(int* out) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *out = c;
            return W4A8_OK;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return W4A8_OK;
}

w4a8::Tuning tuning() {
    w4a8::Tuning t;
    t.force_splits = g_force_splits.load();
    t.force_cl = g_force_cl.load();
    t.ring_bytes = g_ring_bytes.load();
    t.ctas_per_sm = g_ctas_per_sm.load();
    return t;
}

// pair: paired gate/up rows (the gated product in the epilogue).
int plan_for(bool w4, bool fused, int64_t M, int64_t K, int64_t N, w4a8::GemvPlan* pl,
             int sms = 0, bool pair = false) {
    if (sms <= 0) {
        int st = sm_count(&sms);
        if (st != W4A8_OK) return st;
    }
    if (!w4a8::make_gemv_plan(w4, fused, (int)M, K, N, sms, tuning(), pl, pair))
        return fail(W4A8_ERR_SHAPE, "no launch plan for M=%lld K=%lld N=%lld",
                    (long long)M, (long long)K, (long long)N);
    return W4A8_OK;
}

int check_w4a8_shape(int64_t M, int64_t K, int64_t N) {
    if (M < 1 || M > W4A8_MAX_M) return fail(W4A8_ERR_SHAPE, "M=%lld outside [1, %d]", (long long)M, W4A8_MAX_M);
    if (K < 32 || K > 131072 || K % 32) return fail(W4A8_ERR_SHAPE, "K=%lld must be a multiple of 32 in [32, 131072]", (long long)K);
    if (N < 1 || N > 0x7FFFFFFF) return fail(W4A8_ERR_SHAPE, "N=%lld outside [1, 2^31-1]", (long long)N);
    return W4A8_OK;
}

int check_w8a16_shape(int64_t M, int64_t K, int64_t N) {
    if (M < 1 || M > W8A16_MAX_M) return fail(W4A8_ERR_SHAPE, "M=%lld outside [1, %d]", (long long)M, W8A16_MAX_M);
    if (K < 16 || K > 65536 || K % 16) return fail(W4A8_ERR_SHAPE, "K=%lld must be a multiple of 16 in [16, 65536]", (long long)K);
    if (N < 1 || N > 0x7FFFFFFF) return fail(W4A8_ERR_SHAPE, "N=%lld outside [1, 2^31-1]", (long long)N);
    return W4A8_OK;
}

// Tensor-core plan for an M-row W4A8 call, or false when the dp4a path
// serves it (fewer rows than the threshold, or no tensor-core plan).
// group > 0: group-wise scales; the tensor cores take groups that are
// whole 128-code stages of at most 16384 codes, smaller groups stay on the
// dp4a kernel.
bool mma_plan_for(int64_t M, int64_t K, int64_t N, w4a8::MmaPlan* pl, int sms = 0,
                  int64_t group = 0) {
    const int t = g_mma_min_m.load();
    if (M < (t > 0 ? t : group > 0 ? kDefaultMmaMinMGroup : kDefaultMmaMinM)) return false;
    if (group > 0 && (group % 128 || group > 16384)) return false;
    if (sms <= 0 && sm_count(&sms) != W4A8_OK) return false;
    return w4a8::make_mma_plan((int)M, K, N, sms, pl, (int)(group / 64), g_force_splits.load());
}

// Warp-level e4m3 MMA plan for an M-row row-wise W4A8 call, or false when
// another kernel serves it.
bool qmma_plan_for(int64_t M, int64_t K, int64_t N, w4a8::QmmaPlan* pl, int sms = 0) {
    const int t = g_qmma_max_m.load();
    if (t == 1 || M < 2 || M > (t > 1 ? t : kDefaultQmmaMaxM)) return false;
    if (sms <= 0 && sm_count(&sms) != W4A8_OK) return false;
    if (!w4a8::make_qmma_plan((int)M, K, N, sms, pl, g_qmma_r.load(), g_qmma_ops.load() == 1)) return false;
    // default routing: persistent plans on many tiles only
    return t > 1 || (pl->persist && pl->tiles >= kQmmaMinTilesPerSm * sms);
}

// Row-per-thread plan for an M-row W4A8 call, or false when another kernel
// serves it.  gshift >= 0: group-wise scales, groups of 2^gshift codes, on
// the one-thread-per-row kernel from 1 row (rowdot_max_m = 1: never).
bool rowdot_plan_for(int64_t M, int64_t K, int64_t N, w4a8::RowdotPlan* pl, int sms = 0,
                     int gshift = -1) {
    const int t = g_rowdot_max_m.load();
    const int hi = t > 0 ? t : gshift >= 0 ? kDefaultRowdotMaxMGroup : kDefaultRowdotMaxM;
    if (M < (gshift >= 0 ? 1 : 2) || M > hi || (gshift >= 0 && t == 1)) return false;
    if (sms <= 0 && sm_count(&sms) != W4A8_OK) return false;
    // row-wise scales on many tiles: the tensor cores
    if (t == 0 && gshift < 0 && (N + 127) / 128 > 2 * (int64_t)sms) return false;
    const int cl = g_force_cl.load();
    return w4a8::make_rowdot_plan((int)M, K, N, sms, pl, (cl == 2 || cl == 4 || cl == 8) ? cl : 0,
                                  g_ctas_per_sm.load(), gshift, gshift >= 0 ? g_force_splits.load() : 0);
}

// log2 of a group size already checked by check_group.
int log2_group(int64_t group) {
    int s = 0;
    while ((1LL << s) < group) ++s;
    return s;
}

// Group-wise calls that neither single launch serves: the one-thread-per-row
// kernel, one launch per group of up to 8 rows (each streams the weights);
// `full` plans 8 rows, `tail` a shorter last group.
bool group_row_plans(int64_t M, int64_t K, int64_t N, int64_t group, w4a8::RowdotPlan* full,
                     w4a8::RowdotPlan* tail, int sms = 0) {
    if (sms <= 0 && sm_count(&sms) != W4A8_OK) return false;
    const int rg = w4a8::kRowdotMaxM;
    const int gshift = log2_group(group);
    const int fp = g_force_splits.load();
    if (!w4a8::make_rowdot_plan((int)(M < rg ? M : rg), K, N, sms, full, 1, g_ctas_per_sm.load(), gshift, fp))
        return false;
    *tail = *full;
    if (M > rg && M % rg)
        return w4a8::make_rowdot_plan((int)(M % rg), K, N, sms, tail, 1, g_ctas_per_sm.load(), gshift, fp);
    return true;
}

int check_ws(size_t need, void* ws, size_t ws_bytes) {
    if (ws == nullptr || ws_bytes < need)
        return fail(W4A8_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given%s", need,
                    ws ? ws_bytes : (size_t)0, ws ? "" : " (NULL)");
    if (!aligned(ws, 256)) return fail(W4A8_ERR_ALIGN, "workspace must be 256-byte aligned");
    return W4A8_OK;
}

int check_mma_workspace(const w4a8::MmaPlan& pl, void* ws, size_t ws_bytes) {
    if (ws == nullptr || ws_bytes < pl.ws_bytes)
        return fail(W4A8_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given%s", pl.ws_bytes,
                    ws ? ws_bytes : (size_t)0, ws ? "" : " (NULL)");
    if (!aligned(ws, 256)) return fail(W4A8_ERR_ALIGN, "workspace must be 256-byte aligned");
    return W4A8_OK;
}

// One kernel launch handles up to this many activation rows; calls with
// more rows run one launch per group of rows (each streams the weights).
constexpr int kRowGroupW4 = 8;
constexpr int kRowGroupW8 = 4;

// Plans of the row groups of an M-row call: `full` for groups of `rg`
// rows, `tail` for a shorter last group (equal to `full` when there is none).
int plan_row_groups(bool w4, bool fused, int64_t M, int64_t K, int64_t N, int rg,
                    w4a8::GemvPlan* full, w4a8::GemvPlan* tail, int sms = 0) {
    int st = plan_for(w4, fused, M < rg ? M : rg, K, N, full, sms);
    if (st != W4A8_OK) return st;
    *tail = *full;
    if (M > rg && M % rg) st = plan_for(w4, fused, M % rg, K, N, tail, sms);
    return st;
}

// Group-wise scales: `group` a power of two in [32, K] dividing K.
int check_group(int64_t K, int64_t group, int* gshift, int* gld) {
    if (group < 32 || group > K || (group & (group - 1)) || K % group)
        return fail(W4A8_ERR_SHAPE, "group=%lld must be a power of two in [32, K=%lld] dividing K",
                    (long long)group, (long long)K);
    int sh = 0;
    while ((32LL << sh) < group) ++sh;
    *gshift = sh;
    *gld = (int)W4G_SCALE_STRIDE(K, group);
    return W4A8_OK;
}

int check_workspace(const w4a8::GemvPlan& pl, void* ws, size_t ws_bytes) {
    if (pl.ws_bytes == 0) return W4A8_OK;
    if (ws == nullptr || ws_bytes < pl.ws_bytes)
        return fail(W4A8_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given%s", pl.ws_bytes,
                    ws ? ws_bytes : (size_t)0, ws ? "" : " (NULL)");
    if (!aligned(ws, 256)) return fail(W4A8_ERR_ALIGN, "workspace must be 256-byte aligned");
    return W4A8_OK;
}

}  // namespace

cudaError_t w4a8_noalloc_reset(cudaStream_t stream);  // defined with the static scratch below

extern "C" {

int w4_quantize_weights(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* sw, void* stream) {
    if (!W || !Wq || !sw) return fail(W4A8_ERR_NULL, "w4_quantize_weights: NULL pointer");
    if (N < 1 || N > 0x7FFFFFFF) return fail(W4A8_ERR_SHAPE, "N=%lld outside [1, 2^31-1]", (long long)N);
    if (K < 32 || K % 32 || K > (1LL << 30)) return fail(W4A8_ERR_SHAPE, "K=%lld must be a positive multiple of 32", (long long)K);
    if (!aligned(W, 16) || !aligned(Wq, 16) || !aligned(sw, 4))
        return fail(W4A8_ERR_ALIGN, "w4_quantize_weights: W and Wq must be 16-byte aligned");
    cudaError_t e = w4a8::launch_w4_quantize(W, N, K, Wq, sw, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4_quantize_weights launch");
}

int w8_quantize_weights(const float* W, int64_t N, int64_t K, int8_t* Wq8, uint16_t* sw16,
                        void* stream) {
    if (!W || !Wq8 || !sw16) return fail(W4A8_ERR_NULL, "w8_quantize_weights: NULL pointer");
    if (N < 1 || N > 0x7FFFFFFF) return fail(W4A8_ERR_SHAPE, "N=%lld outside [1, 2^31-1]", (long long)N);
    if (K < 16 || K % 16 || K > (1LL << 30)) return fail(W4A8_ERR_SHAPE, "K=%lld must be a positive multiple of 16", (long long)K);
    if (!aligned(W, 16) || !aligned(Wq8, 16) || !aligned(sw16, 2))
        return fail(W4A8_ERR_ALIGN, "w8_quantize_weights: W and Wq8 must be 16-byte aligned");
    cudaError_t e = w4a8::launch_w8_quantize(W, N, K, Wq8, sw16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "w8_quantize_weights launch");
}

int act_quantize_i8(const uint16_t* X, int64_t M, int64_t K, int8_t* Xq, float* sa, void* stream) {
    if (!X || !Xq || !sa) return fail(W4A8_ERR_NULL, "act_quantize_i8: NULL pointer");
    if (M < 1 || M > 65535) return fail(W4A8_ERR_SHAPE, "M=%lld outside [1, 65535]", (long long)M);
    if (K < 1 || K > (1LL << 20) || K % 8) return fail(W4A8_ERR_SHAPE, "K=%lld must be a multiple of 8 in [8, 2^20]", (long long)K);
    if (!aligned(X, 16) || !aligned(Xq, 16) || !aligned(sa, 4))
        return fail(W4A8_ERR_ALIGN, "act_quantize_i8: X and Xq must be 16-byte aligned");
    cudaError_t e = w4a8::launch_act_quantize(X, M, K, Xq, sa, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "act_quantize_i8 launch");
}

size_t w4a8_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    if (check_w4a8_shape(M, K, N) != W4A8_OK) return 0;
    w4a8::QmmaPlan qp;
    if (qmma_plan_for(M, K, N, &qp)) return qp.ws_bytes;
    w4a8::RowdotPlan rp;
    if (rowdot_plan_for(M, K, N, &rp)) return rp.ws_bytes;
    w4a8::MmaPlan mp;
    if (mma_plan_for(M, K, N, &mp)) return mp.ws_bytes;
    w4a8::GemvPlan pf, pt;
    // the fused and unfused kernels share the split plan
    if (plan_row_groups(true, true, M, K, N, kRowGroupW4, &pf, &pt) != W4A8_OK) return 0;
    return pf.ws_bytes > pt.ws_bytes ? pf.ws_bytes : pt.ws_bytes;
}

int w4g_quantize_weights(const float* W, int64_t N, int64_t K, int64_t group, uint8_t* Wq,
                         float* sg, void* stream) {
    if (!W || !Wq || !sg) return fail(W4A8_ERR_NULL, "w4g_quantize_weights: NULL pointer");
    if (N < 1 || N > 0x7FFFFFFF) return fail(W4A8_ERR_SHAPE, "N=%lld outside [1, 2^31-1]", (long long)N);
    if (K < 32 || K % 32 || K > (1LL << 30)) return fail(W4A8_ERR_SHAPE, "K=%lld must be a positive multiple of 32", (long long)K);
    int gshift, gld;
    int st = check_group(K, group, &gshift, &gld);
    if (st != W4A8_OK) return st;
    if (!aligned(W, 16) || !aligned(Wq, 16) || !aligned(sg, 16))
        return fail(W4A8_ERR_ALIGN, "w4g_quantize_weights: W, Wq and sg must be 16-byte aligned");
    cudaError_t e = w4a8::launch_w4g_quantize(W, N, K, (int)group, gld, Wq, sg,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4g_quantize_weights launch");
}

size_t w4a8g_workspace_bytes(int64_t M, int64_t K, int64_t N, int64_t group) {
    if (check_w4a8_shape(M, K, N) != W4A8_OK) return 0;
    int gshift, gld;
    if (check_group(K, group, &gshift, &gld) != W4A8_OK) return 0;
    w4a8::RowdotPlan rp;
    if (rowdot_plan_for(M, K, N, &rp, 0, log2_group(group))) return rp.ws_bytes;
    w4a8::MmaPlan mp;
    if (mma_plan_for(M, K, N, &mp, 0, group)) return mp.ws_bytes;
    w4a8::RowdotPlan pf, pt;
    if (!group_row_plans(M, K, N, group, &pf, &pt)) return 0;
    return pf.ws_bytes > pt.ws_bytes ? pf.ws_bytes : pt.ws_bytes;
}

size_t w8a16_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    if (check_w8a16_shape(M, K, N) != W4A8_OK) return 0;
    w4a8::GemvPlan pf, pt;
    if (plan_row_groups(false, false, M, K, N, kRowGroupW8, &pf, &pt) != W4A8_OK) return 0;
    return pf.ws_bytes > pt.ws_bytes ? pf.ws_bytes : pt.ws_bytes;
}

int w4a8_gemv(const int8_t* Xq, const float* sa, int64_t M, int64_t K, const uint8_t* Wq,
              const float* sw, int64_t N, float* Y, int32_t* acc_out, void* ws, size_t ws_bytes,
              unsigned flags, void* stream) {
    if (!Xq || !sa || !Wq || !sw || !Y) return fail(W4A8_ERR_NULL, "w4a8_gemv: NULL pointer");
    int st = check_w4a8_shape(M, K, N);
    if (st != W4A8_OK) return st;
    if (!aligned(Xq, 16) || !aligned(Wq, 16) || !aligned(Y, 4) || !aligned(sw, 4) ||
        !aligned(sa, 4) || (acc_out && !aligned(acc_out, 4)))
        return fail(W4A8_ERR_ALIGN, "w4a8_gemv: Xq/Wq need 16-byte, Y/sw/sa/acc_out 4-byte alignment");
    w4a8::QmmaPlan qp;
    if (qmma_plan_for(M, K, N, &qp)) {
        if ((st = check_ws(qp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_qmma(qp, nullptr, Xq, sa, (int)M, K, 1, &Wq, &sw, &N, &Y, acc_out,
                                               nullptr, nullptr, ws, flags, static_cast<cudaStream_t>(stream),
                                               qmma_stall_ns());
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_gemv warp-MMA launch");
    }
    w4a8::RowdotPlan rp;
    if (rowdot_plan_for(M, K, N, &rp)) {
        if ((st = check_ws(rp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_rowdot(rp, nullptr, Xq, sa, (int)M, K, 1, &Wq, &sw, &N, &Y,
                                                 acc_out, nullptr, nullptr, ws, flags,
                                                 static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_gemv row-per-thread launch");
    }
    w4a8::MmaPlan mp;
    if (mma_plan_for(M, K, N, &mp)) {
        if ((st = check_mma_workspace(mp, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_mma(mp, nullptr, Xq, sa, (int)M, K, 1, &Wq, &sw, &N, &Y,
                                              acc_out, nullptr, nullptr, ws, flags,
                                              static_cast<cudaStream_t>(stream), 0, nullptr, mma_e4m3());
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_gemv tensor-core launch");
    }
    w4a8::GemvPlan pf, pt;
    if ((st = plan_row_groups(true, true, M, K, N, kRowGroupW4, &pf, &pt)) != W4A8_OK) return st;
    if ((st = check_workspace(pf, ws, ws_bytes)) != W4A8_OK) return st;
    if ((st = check_workspace(pt, ws, ws_bytes)) != W4A8_OK) return st;
    for (int64_t m0 = 0; m0 < M; m0 += kRowGroupW4) {
        const int64_t mg = M - m0 < kRowGroupW4 ? M - m0 : kRowGroupW4;
        cudaError_t e = w4a8::launch_w4a8(mg == kRowGroupW4 || M < kRowGroupW4 ? pf : pt, false,
                                          nullptr, Xq + m0 * K, sa + m0, (int)mg, K, Wq, sw, N,
                                          Y + m0 * N, acc_out ? acc_out + m0 * N : nullptr,
                                          nullptr, nullptr, ws, flags,
                                          static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "w4a8_gemv launch");
    }
    return ok();
}

}  // extern "C"

namespace {
// The L2 prefetch hint of the *_prefetch entry points, passed to the dp4a
// GEMV launch of the call that sets it (this thread only).
thread_local const void* t_prefetch = nullptr;
thread_local int64_t t_prefetch_bytes = 0;

// Sets the hint for one call and clears it afterwards.
struct PrefetchScope {
    PrefetchScope(const void* p, size_t bytes) {
        t_prefetch = p;
        t_prefetch_bytes = p ? (int64_t)bytes : 0;
    }
    ~PrefetchScope() {
        t_prefetch = nullptr;
        t_prefetch_bytes = 0;
    }
};
}  // namespace

extern "C" {

int w4a8_linear(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const float* sw,
                int64_t N, float* Y, int8_t* Xq_out, float* sa_out, int32_t* acc_out, void* ws,
                size_t ws_bytes, unsigned flags, void* stream) {
    if (!X || !Wq || !sw || !Y) return fail(W4A8_ERR_NULL, "w4a8_linear: NULL pointer");
    int st = check_w4a8_shape(M, K, N);
    if (st != W4A8_OK) return st;
    if (!aligned(X, 16) || !aligned(Wq, 16) || !aligned(Y, 4) || !aligned(sw, 4) ||
        (Xq_out && !aligned(Xq_out, 16)) || (sa_out && !aligned(sa_out, 4)) ||
        (acc_out && !aligned(acc_out, 4)))
        return fail(W4A8_ERR_ALIGN, "w4a8_linear: X/Wq/Xq_out need 16-byte, Y/sw/sa_out/acc_out 4-byte alignment");
    w4a8::QmmaPlan qp;
    if (qmma_plan_for(M, K, N, &qp)) {
        if ((st = check_ws(qp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_qmma(qp, X, nullptr, nullptr, (int)M, K, 1, &Wq, &sw, &N, &Y,
                                               acc_out, Xq_out, sa_out, ws, flags,
                                               static_cast<cudaStream_t>(stream), qmma_stall_ns());
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear warp-MMA launch");
    }
    w4a8::RowdotPlan rp;
    if (rowdot_plan_for(M, K, N, &rp)) {
        if ((st = check_ws(rp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_rowdot(rp, X, nullptr, nullptr, (int)M, K, 1, &Wq, &sw, &N,
                                                 &Y, acc_out, Xq_out, sa_out, ws, flags,
                                                 static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear row-per-thread launch");
    }
    w4a8::MmaPlan mp;
    if (mma_plan_for(M, K, N, &mp)) {
        if ((st = check_mma_workspace(mp, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_mma(mp, X, nullptr, nullptr, (int)M, K, 1, &Wq, &sw, &N,
                                              &Y, acc_out, Xq_out, sa_out, ws, flags,
                                              static_cast<cudaStream_t>(stream), 0, nullptr, mma_e4m3());
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear tensor-core launch");
    }
    w4a8::GemvPlan pf, pt;
    if ((st = plan_row_groups(true, true, M, K, N, kRowGroupW4, &pf, &pt)) != W4A8_OK) return st;
    if ((st = check_workspace(pf, ws, ws_bytes)) != W4A8_OK) return st;
    if ((st = check_workspace(pt, ws, ws_bytes)) != W4A8_OK) return st;
    for (int64_t m0 = 0; m0 < M; m0 += kRowGroupW4) {
        const int64_t mg = M - m0 < kRowGroupW4 ? M - m0 : kRowGroupW4;
        cudaError_t e = w4a8::launch_w4a8(mg == kRowGroupW4 || M < kRowGroupW4 ? pf : pt, true,
                                          X + m0 * K, nullptr, nullptr, (int)mg, K, Wq, sw, N,
                                          Y + m0 * N, acc_out ? acc_out + m0 * N : nullptr,
                                          Xq_out ? Xq_out + m0 * K : nullptr,
                                          sa_out ? sa_out + m0 : nullptr, ws, flags,
                                          static_cast<cudaStream_t>(stream), t_prefetch, t_prefetch_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "w4a8_linear launch");
    }
    return ok();
}

int w4a8_linear_grouped(const uint16_t* X, int64_t M, int64_t K, int G, const uint8_t* const* Wq,
                        const float* const* sw, const int64_t* N, float* const* Y, void* ws,
                        size_t ws_bytes, unsigned flags, void* stream) {
    if (!X || !Wq || !sw || !N || !Y) return fail(W4A8_ERR_NULL, "w4a8_linear_grouped: NULL pointer");
    if (G < 1 || G > W4A8_MAX_GROUP)
        return fail(W4A8_ERR_SHAPE, "G=%d outside [1, %d]", G, W4A8_MAX_GROUP);
    int64_t total = 0;
    for (int g = 0; g < G; ++g) {
        if (!Wq[g] || !sw[g] || !Y[g]) return fail(W4A8_ERR_NULL, "w4a8_linear_grouped: NULL pointer in group %d", g);
        if (N[g] < 1) return fail(W4A8_ERR_SHAPE, "N[%d]=%lld < 1", g, (long long)N[g]);
        if (!aligned(Wq[g], 16) || !aligned(sw[g], 4) || !aligned(Y[g], 4))
            return fail(W4A8_ERR_ALIGN, "w4a8_linear_grouped: Wq[%d] needs 16-byte, sw/Y 4-byte alignment", g);
        total += N[g];
    }
    int st = check_w4a8_shape(M, K, total);
    if (st != W4A8_OK) return st;
    if (!aligned(X, 16)) return fail(W4A8_ERR_ALIGN, "w4a8_linear_grouped: X needs 16-byte alignment");
    w4a8::QmmaPlan qp;
    if (qmma_plan_for(M, K, total, &qp)) {
        // one plan per matrix inside; the workspace bound covers every N[g] <= total
        for (int g = 0; g < G; ++g) {
            w4a8::QmmaPlan pg;
            if (!w4a8::make_qmma_plan((int)M, K, N[g], qp.sms, &pg, qp.R, qp.h16 != 0) || pg.ws_bytes > qp.ws_bytes)
                return fail(W4A8_ERR_SHAPE, "no warp-MMA plan for group %d", g);
        }
        if ((st = check_ws(qp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_qmma(qp, X, nullptr, nullptr, (int)M, K, G, Wq, sw, N, Y, nullptr,
                                               nullptr, nullptr, ws, flags, static_cast<cudaStream_t>(stream),
                                               qmma_stall_ns());
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear_grouped warp-MMA launch");
    }
    w4a8::RowdotPlan rp;
    if (rowdot_plan_for(M, K, total, &rp)) {
        // one plan per matrix inside; the workspace bound covers every N[g] <= total
        for (int g = 0; g < G; ++g) {
            w4a8::RowdotPlan pg;
            if (!w4a8::make_rowdot_plan((int)M, K, N[g], rp.sms, &pg, rp.tpr, rp.cps) ||
                pg.ws_bytes > rp.ws_bytes)
                return fail(W4A8_ERR_SHAPE, "no row-per-thread plan for group %d", g);
        }
        if ((st = check_ws(rp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_rowdot(rp, X, nullptr, nullptr, (int)M, K, G, Wq, sw, N, Y,
                                                 nullptr, nullptr, nullptr, ws, flags,
                                                 static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear_grouped row-per-thread launch");
    }
    w4a8::MmaPlan mp;
    if (mma_plan_for(M, K, total, &mp)) {
        // one plan per matrix inside; the workspace bound covers every N[g] <= total
        for (int g = 0; g < G; ++g) {
            w4a8::MmaPlan pg;
            if (!w4a8::make_mma_plan((int)M, K, N[g], mp.sms, &pg, 0, mp.force_p) || pg.ws_bytes > mp.ws_bytes)
                return fail(W4A8_ERR_SHAPE, "no tensor-core plan for group %d", g);
        }
        if ((st = check_mma_workspace(mp, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_mma(mp, X, nullptr, nullptr, (int)M, K, G, Wq, sw, N, Y,
                                              nullptr, nullptr, nullptr, ws, flags,
                                              static_cast<cudaStream_t>(stream), 0, nullptr, mma_e4m3());
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear_grouped tensor-core launch");
    }
    w4a8::GemvPlan pf, pt;
    if ((st = plan_row_groups(true, true, M, K, total, kRowGroupW4, &pf, &pt)) != W4A8_OK) return st;
    if ((st = check_workspace(pf, ws, ws_bytes)) != W4A8_OK) return st;
    if ((st = check_workspace(pt, ws, ws_bytes)) != W4A8_OK) return st;
    float* Yg[W4A8_MAX_GROUP];
    for (int64_t m0 = 0; m0 < M; m0 += kRowGroupW4) {
        const int64_t mg = M - m0 < kRowGroupW4 ? M - m0 : kRowGroupW4;
        for (int g = 0; g < G; ++g) Yg[g] = Y[g] + m0 * N[g];
        cudaError_t e = w4a8::launch_w4a8_grouped(mg == kRowGroupW4 || M < kRowGroupW4 ? pf : pt,
                                                  X + m0 * K, (int)mg, K, G, Wq, sw, N, Yg, ws,
                                                  flags, static_cast<cudaStream_t>(stream), t_prefetch,
                                                  t_prefetch_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "w4a8_linear_grouped launch");
    }
    return ok();
}

}  // extern "C"

namespace {

// Shared body of the group-scale entry points: X (fused) or Xq + sa.
int w4a8g_run(const char* name, const uint16_t* X, const int8_t* Xq, const float* sa, int64_t M,
              int64_t K, int64_t group, int G, const uint8_t* const* Wq, const float* const* sg,
              const int64_t* N, float* const* Y, int8_t* Xq_out, float* sa_out, void* ws,
              size_t ws_bytes, unsigned flags, void* stream) {
    if (G < 1 || G > W4A8_MAX_GROUP)
        return fail(W4A8_ERR_SHAPE, "%s: G=%d outside [1, %d]", name, G, W4A8_MAX_GROUP);
    int64_t total = 0;
    for (int g = 0; g < G; ++g) {
        if (!Wq[g] || !sg[g] || !Y[g]) return fail(W4A8_ERR_NULL, "%s: NULL pointer in group %d", name, g);
        if (N[g] < 1) return fail(W4A8_ERR_SHAPE, "%s: N[%d]=%lld < 1", name, g, (long long)N[g]);
        if (!aligned(Wq[g], 16) || !aligned(sg[g], 16) || !aligned(Y[g], 4))
            return fail(W4A8_ERR_ALIGN, "%s: Wq and sg need 16-byte, Y 4-byte alignment", name);
        total += N[g];
    }
    int st = check_w4a8_shape(M, K, total);
    if (st != W4A8_OK) return st;
    int gshift, gld;
    if ((st = check_group(K, group, &gshift, &gld)) != W4A8_OK) return st;
    if ((X && !aligned(X, 16)) || (Xq && !aligned(Xq, 16)) || (sa && !aligned(sa, 4)) ||
        (Xq_out && !aligned(Xq_out, 16)) || (sa_out && !aligned(sa_out, 4)))
        return fail(W4A8_ERR_ALIGN, "%s: X/Xq/Xq_out need 16-byte, sa/sa_out 4-byte alignment", name);
    w4a8::RowdotPlan rp;
    if (rowdot_plan_for(M, K, total, &rp, 0, log2_group(group))) {
        // one launch for every matrix; its plan (whole tiles per matrix) fits this workspace
        if ((st = check_ws(rp.ws_bytes, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_rowdot(rp, X, Xq, sa, (int)M, K, G, Wq, nullptr, N, Y, nullptr,
                                                 Xq_out, sa_out, ws, flags,
                                                 static_cast<cudaStream_t>(stream), (int)group, sg);
        return e == cudaSuccess ? ok() : cuda_fail(e, name);
    }
    w4a8::MmaPlan mp;
    if (mma_plan_for(M, K, total, &mp, 0, group)) {
        // one plan per matrix inside; the workspace bound covers every N[g] <= total
        for (int g = 0; g < G; ++g) {
            w4a8::MmaPlan pg;
            if (!w4a8::make_mma_plan((int)M, K, N[g], mp.sms, &pg, (int)(group / 64), mp.force_p) ||
                pg.ws_bytes > mp.ws_bytes)
                return fail(W4A8_ERR_SHAPE, "%s: no tensor-core plan for group %d", name, g);
        }
        if ((st = check_mma_workspace(mp, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_mma(mp, X, Xq, sa, (int)M, K, G, Wq, nullptr, N, Y, nullptr,
                                              Xq_out, sa_out, ws, flags,
                                              static_cast<cudaStream_t>(stream), (int)group, sg);
        return e == cudaSuccess ? ok() : cuda_fail(e, name);
    }
    w4a8::RowdotPlan pf, pt;
    if (!group_row_plans(M, K, total, group, &pf, &pt))
        return fail(W4A8_ERR_SHAPE, "%s: no launch plan for M=%lld K=%lld N=%lld", name, (long long)M,
                    (long long)K, (long long)total);
    if ((st = check_ws(pf.ws_bytes > pt.ws_bytes ? pf.ws_bytes : pt.ws_bytes, ws, ws_bytes)) != W4A8_OK)
        return st;
    const int rg = w4a8::kRowdotMaxM;
    float* Yg[W4A8_MAX_GROUP];
    for (int64_t m0 = 0; m0 < M; m0 += rg) {
        const int64_t mg = M - m0 < rg ? M - m0 : rg;
        for (int g = 0; g < G; ++g) Yg[g] = Y[g] + m0 * N[g];
        cudaError_t e = w4a8::launch_w4a8_rowdot(
            mg == rg || M < rg ? pf : pt, X ? X + m0 * K : nullptr, Xq ? Xq + m0 * K : nullptr,
            sa ? sa + m0 : nullptr, (int)mg, K, G, Wq, nullptr, N, Yg, nullptr,
            Xq_out ? Xq_out + m0 * K : nullptr, sa_out ? sa_out + m0 : nullptr, ws, flags,
            static_cast<cudaStream_t>(stream), (int)group, sg);
        if (e != cudaSuccess) return cuda_fail(e, name);
    }
    return ok();
}

}  // namespace

extern "C" {

int w4a8g_gemv(const int8_t* Xq, const float* sa, int64_t M, int64_t K, int64_t group,
               const uint8_t* Wq, const float* sg, int64_t N, float* Y, void* ws,
               size_t ws_bytes, unsigned flags, void* stream) {
    if (!Xq || !sa || !Wq || !sg || !Y) return fail(W4A8_ERR_NULL, "w4a8g_gemv: NULL pointer");
    return w4a8g_run("w4a8g_gemv", nullptr, Xq, sa, M, K, group, 1, &Wq, &sg, &N, &Y, nullptr,
                     nullptr, ws, ws_bytes, flags, stream);
}

int w4a8g_linear(const uint16_t* X, int64_t M, int64_t K, int64_t group, const uint8_t* Wq,
                 const float* sg, int64_t N, float* Y, int8_t* Xq_out, float* sa_out, void* ws,
                 size_t ws_bytes, unsigned flags, void* stream) {
    if (!X || !Wq || !sg || !Y) return fail(W4A8_ERR_NULL, "w4a8g_linear: NULL pointer");
    return w4a8g_run("w4a8g_linear", X, nullptr, nullptr, M, K, group, 1, &Wq, &sg, &N, &Y,
                     Xq_out, sa_out, ws, ws_bytes, flags, stream);
}

int w4a8g_linear_grouped(const uint16_t* X, int64_t M, int64_t K, int64_t group, int G,
                         const uint8_t* const* Wq, const float* const* sg, const int64_t* N,
                         float* const* Y, void* ws, size_t ws_bytes, unsigned flags,
                         void* stream) {
    if (!X || !Wq || !sg || !N || !Y) return fail(W4A8_ERR_NULL, "w4a8g_linear_grouped: NULL pointer");
    return w4a8g_run("w4a8g_linear_grouped", X, nullptr, nullptr, M, K, group, G, Wq, sg, N, Y,
                     nullptr, nullptr, ws, ws_bytes, flags, stream);
}

int w8a16_gemv(const uint16_t* X, int64_t M, int64_t K, const int8_t* Wq8, const uint16_t* sw16,
               int64_t N, float* Y, void* ws, size_t ws_bytes, unsigned flags, void* stream) {
    if (!X || !Wq8 || !sw16 || !Y) return fail(W4A8_ERR_NULL, "w8a16_gemv: NULL pointer");
    int st = check_w8a16_shape(M, K, N);
    if (st != W4A8_OK) return st;
    if (!aligned(X, 16) || !aligned(Wq8, 16) || !aligned(Y, 4) || !aligned(sw16, 2))
        return fail(W4A8_ERR_ALIGN, "w8a16_gemv: X/Wq8 need 16-byte, Y 4-byte alignment");
    w4a8::GemvPlan pf, pt;
    if ((st = plan_row_groups(false, false, M, K, N, kRowGroupW8, &pf, &pt)) != W4A8_OK) return st;
    if ((st = check_workspace(pf, ws, ws_bytes)) != W4A8_OK) return st;
    if ((st = check_workspace(pt, ws, ws_bytes)) != W4A8_OK) return st;
    for (int64_t m0 = 0; m0 < M; m0 += kRowGroupW8) {
        const int64_t mg = M - m0 < kRowGroupW8 ? M - m0 : kRowGroupW8;
        cudaError_t e = w4a8::launch_w8a16(mg == kRowGroupW8 || M < kRowGroupW8 ? pf : pt,
                                           X + m0 * K, (int)mg, K, Wq8, sw16, N, Y + m0 * N, ws,
                                           flags, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "w8a16_gemv launch");
    }
    return ok();
}

int index_softmax_lut(int b, double c, uint8_t* lut) {
    if (!lut) return fail(W4A8_ERR_NULL, "index_softmax_lut: NULL pointer");
    if (b < 1 || b > 8 || !(c > 0.0) || !(c < 1e300))
        return fail(W4A8_ERR_SHAPE, "index_softmax_lut: need 1 <= b <= 8 and c > 0");
    w4a8::isx_build_lut(b, c, lut);
    return ok();
}

int64_t index_softmax_c_int(double c, int64_t d, float s_q, float s_k) {
    if (!(c > 0.0) || d < 1 || !(s_q > 0.f) || !(s_k > 0.f)) return -1;
    const double v = c * std::sqrt((double)d) / ((double)s_q * (double)s_k);
    if (!(v < 2147483647.0)) return -1;
    return w4a8::isx_c_int(c, d, s_q, s_k);
}

int index_softmax_u8(const int32_t* A, int64_t rows, int64_t cols, int64_t c_int, int b,
                     const uint8_t* lut, uint8_t* P, void* stream) {
    if (!A || !lut || !P) return fail(W4A8_ERR_NULL, "index_softmax_u8: NULL pointer");
    if (rows < 1 || rows > 0x7FFFFFFF)
        return fail(W4A8_ERR_SHAPE, "rows=%lld outside [1, 2^31-1]", (long long)rows);
    if (cols < 1 || cols > ISX_MAX_COLS)
        return fail(W4A8_ERR_SHAPE, "cols=%lld outside [1, %d]", (long long)cols, ISX_MAX_COLS);
    if (c_int < 0 || c_int > 0x7FFFFFFF)
        return fail(W4A8_ERR_SHAPE, "c_int=%lld outside [0, 2^31-1]", (long long)c_int);
    if (b < 1 || b > 8) return fail(W4A8_ERR_SHAPE, "b=%d outside [1, 8]", b);
    if (lut[0] < 1) return fail(W4A8_ERR_SHAPE, "lut[0] must be at least 1 (row sums stay positive)");
    if (!aligned(A, 4)) return fail(W4A8_ERR_ALIGN, "index_softmax_u8: A needs 4-byte alignment");
    uint32_t thr[w4a8::kIsxMaxEntries + 1];
    w4a8::isx_thresholds((uint32_t)c_int, b, thr);
    cudaError_t e = w4a8::launch_index_softmax(A, rows, cols, (uint32_t)c_int, b, lut, thr, P,
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "index_softmax_u8 launch");
}

const char* w4a8_last_error(void) { return g_last_error.c_str(); }

int w4a8_device_error(unsigned* flags, void* stream) {
    if (!flags) return fail(W4A8_ERR_NULL, "w4a8_device_error: NULL pointer");
    *flags = 0;
    cudaError_t e = w4a8::read_and_clear_device_error(flags, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = w4a8::read_and_clear_mma_error(flags, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = w4a8::read_and_clear_rowdot_error(flags, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = w4a8::read_and_clear_qmma_error(flags, static_cast<cudaStream_t>(stream));
    // a wait that gave up may leave split-K arrival counters non-zero; the
    // static scratch of w4a8_linear_noalloc is cleared here (caller-owned
    // workspaces must be re-zeroed by the caller)
    if (e == cudaSuccess && *flags != 0) {
        e = w4a8_noalloc_reset(static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_device_error");
}

int w4a8_set_tuning(const w4a8_tuning_t* t) {
    if (t == nullptr) {
        g_force_splits = 0;
        g_force_cl = 0;
        g_ring_bytes = 0;
        g_ctas_per_sm = 0;
        g_mma_min_m = 0;
        g_rowdot_max_m = 0;
        g_mma_e4m3 = 0;
        g_qmma_max_m = 0;
        g_qmma_r = 0;
        g_stall_test_us = 0;
        g_qmma_ops = 0;
        return ok();
    }
    if (t->force_splits < 0 || t->force_splits > 16)
        return fail(W4A8_ERR_SHAPE, "force_splits must be in [0, 16]");
    if (t->force_threads_per_row < 0 || t->force_threads_per_row > 256 ||
        (t->force_threads_per_row & (t->force_threads_per_row - 1)))
        return fail(W4A8_ERR_SHAPE, "force_threads_per_row must be 0 or a power of two <= 256");
    if (t->ring_bytes < 0 || t->ring_bytes > 200 * 1024)
        return fail(W4A8_ERR_SHAPE, "ring_bytes must be in [0, 204800]");
    if (t->ctas_per_sm < 0 || t->ctas_per_sm > 4)
        return fail(W4A8_ERR_SHAPE, "ctas_per_sm must be in [0, 4]");
    g_force_splits = t->force_splits;
    g_force_cl = t->force_threads_per_row;
    g_ring_bytes = t->ring_bytes;
    if (t->mma_min_m != 0 && (t->mma_min_m < 2 || t->mma_min_m > 65))
        return fail(W4A8_ERR_SHAPE, "mma_min_m must be 0 or in [2, 65]");
    if (t->rowdot_max_m < 0 || t->rowdot_max_m > w4a8::kRowdotMaxM)
        return fail(W4A8_ERR_SHAPE, "rowdot_max_m must be in [0, %d]", w4a8::kRowdotMaxM);
    g_ctas_per_sm = t->ctas_per_sm;
    g_mma_min_m = t->mma_min_m;
    g_rowdot_max_m = t->rowdot_max_m;
    if (t->mma_e4m3 < 0 || t->mma_e4m3 > 2) return fail(W4A8_ERR_SHAPE, "mma_e4m3 must be 0, 1 or 2");
    g_mma_e4m3 = t->mma_e4m3;
    if (t->qmma_max_m < 0 || t->qmma_max_m > w4a8::kQmmaMaxM)
        return fail(W4A8_ERR_SHAPE, "qmma_max_m must be in [0, %d]", w4a8::kQmmaMaxM);
    g_qmma_max_m = t->qmma_max_m;
    if (t->qmma_tiles_per_warp != 0 && t->qmma_tiles_per_warp != 1 && t->qmma_tiles_per_warp != 2 &&
        t->qmma_tiles_per_warp != 4)
        return fail(W4A8_ERR_SHAPE, "qmma_tiles_per_warp must be 0, 1, 2 or 4");
    g_qmma_r = t->qmma_tiles_per_warp;
    if (t->stall_test_us < 0 || t->stall_test_us > 1000000)
        return fail(W4A8_ERR_SHAPE, "stall_test_us must be in [0, 1000000]");
    g_stall_test_us = t->stall_test_us;
    if (t->qmma_operands < 0 || t->qmma_operands > 2)
        return fail(W4A8_ERR_SHAPE, "qmma_operands must be 0, 1 or 2");
    g_qmma_ops = t->qmma_operands;
    return ok();
}

int w4a8_plan_info(int64_t M, int64_t K, int64_t N, int w8a16, int num_sms, int* info,
                   int n_info) {
    if (!info) return fail(W4A8_ERR_NULL, "w4a8_plan_info: NULL pointer");
    int st = w8a16 ? check_w8a16_shape(M, K, N) : check_w4a8_shape(M, K, N);
    if (st != W4A8_OK) return st;
    if (!w8a16) {
        w4a8::QmmaPlan qp;
        if (qmma_plan_for(M, K, N, &qp, num_sms)) {
            const int ws = qp.ws_bytes > 0x7FFFFFFF ? 0x7FFFFFFF : (int)qp.ws_bytes;
            const int v[] = {qp.P, qp.R, (qp.h16 ? 8 : 4) * qp.NT, 128, qp.tiles, qp.grid, 128, qp.NS, qp.stage_bytes,
                             qp.smem, ws, 3};
            for (int k = 0; k < n_info && k < (int)(sizeof(v) / sizeof(v[0])); ++k) info[k] = v[k];
            return ok();
        }
        w4a8::RowdotPlan rp;
        if (rowdot_plan_for(M, K, N, &rp, num_sms)) {
            const int ws = rp.ws_bytes > 0x7FFFFFFF ? 0x7FFFFFFF : (int)rp.ws_bytes;
            const int v[] = {rp.P, rp.tpr, rp.MT, 128, rp.tiles, rp.grid, 128, rp.NS, 16384,
                             rp.smem, ws, 2};
            for (int k = 0; k < n_info && k < (int)(sizeof(v) / sizeof(v[0])); ++k) info[k] = v[k];
            return ok();
        }
        w4a8::MmaPlan mp;
        if (mma_plan_for(M, K, N, &mp, num_sms)) {
            const int ws = mp.ws_bytes > 0x7FFFFFFF ? 0x7FFFFFFF : (int)mp.ws_bytes;
            const int v[] = {mp.P, 0, mp.BN, 128, mp.tiles, mp.grid, 128, mp.stages, mp.stage_bytes,
                             mp.smem, ws, 1};
            for (int k = 0; k < n_info && k < (int)(sizeof(v) / sizeof(v[0])); ++k) info[k] = v[k];
            return ok();
        }
    }
    // the plan of the first row group; workspace for the whole call
    w4a8::GemvPlan pl, pt;
    if ((st = plan_row_groups(!w8a16, !w8a16, M, K, N, w8a16 ? kRowGroupW8 : kRowGroupW4, &pl,
                              &pt, num_sms)) != W4A8_OK)
        return st;
    const size_t wsb = pl.ws_bytes > pt.ws_bytes ? pl.ws_bytes : pt.ws_bytes;
    const int ws = wsb > 0x7FFFFFFF ? 0x7FFFFFFF : (int)wsb;
    const int v[] = {pl.P, pl.Cl, pl.S, pl.Rl, pl.Gs, pl.grid, pl.rows_max, pl.NS,
                     pl.stage_stride, pl.smem, ws, 0};
    for (int k = 0; k < n_info && k < (int)(sizeof(v) / sizeof(v[0])); ++k) info[k] = v[k];
    return ok();
}

int w4a8g_plan_info(int64_t M, int64_t K, int64_t N, int64_t group, int num_sms, int* info,
                    int n_info) {
    if (!info) return fail(W4A8_ERR_NULL, "w4a8g_plan_info: NULL pointer");
    int st = check_w4a8_shape(M, K, N);
    if (st != W4A8_OK) return st;
    int gshift, gld;
    if ((st = check_group(K, group, &gshift, &gld)) != W4A8_OK) return st;
    // the last two entries: the fold chunks of the group-scale contract
    // (count, codes per chunk)
    const int64_t chunk = group > 1024 ? group : 1024;
    const int nch = (int)((K + chunk - 1) / chunk);
    w4a8::RowdotPlan rp, rt;
    const bool single = rowdot_plan_for(M, K, N, &rp, num_sms, log2_group(group));
    w4a8::MmaPlan mp;
    if (!single && mma_plan_for(M, K, N, &mp, num_sms, group)) {
        const int ws = mp.ws_bytes > 0x7FFFFFFF ? 0x7FFFFFFF : (int)mp.ws_bytes;
        const int v[] = {mp.P, 0, mp.BN, 128, mp.tiles, mp.grid, 128, mp.stages, mp.stage_bytes,
                         mp.smem, ws, 1, nch, (int)chunk};
        for (int k = 0; k < n_info && k < (int)(sizeof(v) / sizeof(v[0])); ++k) info[k] = v[k];
        return ok();
    }
    // one launch, or the plan of the first group of 8 rows; workspace for the whole call
    if (!single && !group_row_plans(M, K, N, group, &rp, &rt, num_sms))
        return fail(W4A8_ERR_SHAPE, "no launch plan for M=%lld K=%lld N=%lld", (long long)M, (long long)K,
                    (long long)N);
    const size_t wsb = single ? rp.ws_bytes : rp.ws_bytes > rt.ws_bytes ? rp.ws_bytes : rt.ws_bytes;
    const int ws = wsb > 0x7FFFFFFF ? 0x7FFFFFFF : (int)wsb;
    const int v[] = {rp.P, rp.tpr, rp.MT, 128, rp.tiles, rp.grid, 128, rp.NS, 16384,
                     rp.smem, ws, 2, nch, (int)chunk};
    for (int k = 0; k < n_info && k < (int)(sizeof(v) / sizeof(v[0])); ++k) info[k] = v[k];
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The MLP's gated product: gate/up projections with silu(gate) * up in the
// epilogue, the stand-alone product, and the row interleaving it reads.
// ---------------------------------------------------------------------------

extern "C" {

size_t w4a8_gate_up_silu_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    if (N < 1 || N > 0x3FFFFFFF || check_w4a8_shape(M, K, 2 * N) != W4A8_OK) return 0;
    if (M > 1) return w4a8_workspace_bytes(M, K, 2 * N);
    w4a8::GemvPlan pl;
    if (plan_for(true, true, 1, K, 2 * N, &pl, 0, true) != W4A8_OK) return 0;
    return pl.ws_bytes;
}

int w4a8_gate_up_silu(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq_gu, const float* sw_gu,
                      int64_t N, float* Y_gu, uint16_t* H, void* ws, size_t ws_bytes, unsigned flags,
                      void* stream) {
    if (!X || !Wq_gu || !sw_gu || !Y_gu || !H) return fail(W4A8_ERR_NULL, "w4a8_gate_up_silu: NULL pointer");
    if (N < 1 || N > 0x3FFFFFFF) return fail(W4A8_ERR_SHAPE, "N=%lld outside [1, 2^30-1]", (long long)N);
    int st = check_w4a8_shape(M, K, 2 * N);
    if (st != W4A8_OK) return st;
    if (!aligned(X, 16) || !aligned(Wq_gu, 16) || !aligned(Y_gu, 4) || !aligned(sw_gu, 4) || !aligned(H, 2))
        return fail(W4A8_ERR_ALIGN, "w4a8_gate_up_silu: X/Wq need 16-byte, Y/sw 4-byte, H 2-byte alignment");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 1) {
        w4a8::GemvPlan pl;
        if ((st = plan_for(true, true, 1, K, 2 * N, &pl, 0, true)) != W4A8_OK) return st;
        if ((st = check_workspace(pl, ws, ws_bytes)) != W4A8_OK) return st;
        cudaError_t e = w4a8::launch_w4a8_silu(pl, X, 1, K, Wq_gu, sw_gu, 2 * N, Y_gu, H, ws, flags, s);
        return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_gate_up_silu launch");
    }
    // batches: the linear on the interleaved matrix, then the product as a
    // launch of its own
    if ((st = w4a8_linear(X, M, K, Wq_gu, sw_gu, 2 * N, Y_gu, nullptr, nullptr, nullptr, ws, ws_bytes, flags,
                          stream)) != W4A8_OK)
        return st;
    cudaError_t e = w4a8::launch_silu_mul(Y_gu, Y_gu + 1, N, M, 2, 2 * N, H, flags, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_gate_up_silu product launch");
}

int w4a8_silu_mul(const float* g, const float* u, int64_t M, int64_t N, uint16_t* H, unsigned flags,
                  void* stream) {
    if (!g || !u || !H) return fail(W4A8_ERR_NULL, "w4a8_silu_mul: NULL pointer");
    if (M < 1 || M > 65535 || N < 1 || N > 0x7FFFFFFF)
        return fail(W4A8_ERR_SHAPE, "w4a8_silu_mul: M=%lld, N=%lld out of range", (long long)M, (long long)N);
    if (!aligned(g, 4) || !aligned(u, 4) || !aligned(H, 2))
        return fail(W4A8_ERR_ALIGN, "w4a8_silu_mul: g/u need 4-byte, H 2-byte alignment");
    cudaError_t e = w4a8::launch_silu_mul(g, u, N, M, 1, N, H, flags, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_silu_mul launch");
}

int w4_interleave_rows(const uint8_t* Wq_a, const float* sw_a, const uint8_t* Wq_b, const float* sw_b,
                       int64_t N, int64_t K, uint8_t* Wq_out, float* sw_out, void* stream) {
    if (!Wq_a || !sw_a || !Wq_b || !sw_b || !Wq_out || !sw_out)
        return fail(W4A8_ERR_NULL, "w4_interleave_rows: NULL pointer");
    if (N < 1 || N > 0x3FFFFFFF || K < 32 || K % 32 || K > (1LL << 30))
        return fail(W4A8_ERR_SHAPE, "w4_interleave_rows: N=%lld, K=%lld out of range", (long long)N, (long long)K);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t rb = (size_t)(K / 2);
    cudaError_t e = cudaMemcpy2DAsync(Wq_out, 2 * rb, Wq_a, rb, rb, (size_t)N, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(Wq_out + rb, 2 * rb, Wq_b, rb, rb, (size_t)N, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(sw_out, 8, sw_a, 4, 4, (size_t)N, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(sw_out + 1, 8, sw_b, 4, 4, (size_t)N, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4_interleave_rows copy");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// w4a8_linear_noalloc: the fused linear with its split-K scratch in a static
// device array, for callers that cannot provide workspace memory.
// ---------------------------------------------------------------------------

namespace {

// Scratch of the split-K kernel: 4096 bytes of arrival counters, then the
// int32 partial sums.  Every GPU that loads this library holds it until exit.
// A __device__ array starts zeroed when the library's device code is loaded
// on a device, and every completed call leaves the counters at zero.
constexpr size_t kNoAllocScratchBytes = W4A8_NOALLOC_SCRATCH;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the current device's scratch array.  In host code the
// array's name is only a stand-in, never a device address, so it is looked
// up on every call (the lookup allocates nothing and stays right if the
// context, and with it the array, is ever created anew).
int noalloc_scratch(void** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    *out = p;
    return W4A8_OK;
}

}  // namespace

// Clears the static scratch's arrival counters on `stream` (after a call
// that gave up on a wait they may be left non-zero).
cudaError_t w4a8_noalloc_reset(cudaStream_t stream) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(p, 0, w4a8::kTicketBytes, stream);
}

extern "C" int w4a8_linear_noalloc(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                                   const float* sw, int64_t N, float* Y, unsigned flags,
                                   void* stream) {
    if (!X || !Wq || !sw || !Y) return fail(W4A8_ERR_NULL, "w4a8_linear_noalloc: NULL pointer");
    int st = check_w4a8_shape(M, K, N);
    if (st != W4A8_OK) return st;
    if (M > kRowGroupW4)
        return fail(W4A8_ERR_SHAPE, "w4a8_linear_noalloc: M=%lld outside [1, %d]", (long long)M, kRowGroupW4);
    if (!aligned(X, 16) || !aligned(Wq, 16) || !aligned(Y, 4) || !aligned(sw, 4))
        return fail(W4A8_ERR_ALIGN, "w4a8_linear_noalloc: X/Wq need 16-byte, Y/sw 4-byte alignment");
    // the kernel w4a8_linear picks, when its workspace fits the scratch
    const size_t need = w4a8_workspace_bytes(M, K, N);
    if (need > 0 && need <= kNoAllocScratchBytes) {
        void* scratch = nullptr;
        if ((st = noalloc_scratch(&scratch)) != W4A8_OK) return st;
        return w4a8_linear(X, M, K, Wq, sw, N, Y, nullptr, nullptr, nullptr, scratch, kNoAllocScratchBytes,
                           flags, stream);
    }
    // else the dp4a GEMV, one launch, when its split-K scratch fits
    w4a8::GemvPlan pl;
    if ((st = plan_for(true, true, M, K, N, &pl)) != W4A8_OK) return st;
    if (pl.ws_bytes > kNoAllocScratchBytes)
        return fail(W4A8_ERR_WORKSPACE,
                    "w4a8_linear_noalloc: this shape needs %zu bytes of split-K scratch, more than "
                    "the %zu-byte static scratch; use w4a8_linear with a workspace",
                    pl.ws_bytes, kNoAllocScratchBytes);
    void* scratch = nullptr;
    if (pl.ws_bytes > 0 && (st = noalloc_scratch(&scratch)) != W4A8_OK) return st;
    cudaError_t e = w4a8::launch_w4a8(pl, true, X, nullptr, nullptr, (int)M, K, Wq, sw, N, Y,
                                      nullptr, nullptr, nullptr, scratch, flags,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ok() : cuda_fail(e, "w4a8_linear_noalloc launch");
}

// ---------------------------------------------------------------------------
// The linear with an L2 prefetch hint for the next launch's weights.
// ---------------------------------------------------------------------------

extern "C" {

int w4a8_linear_prefetch(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const float* sw,
                         int64_t N, float* Y, void* ws, size_t ws_bytes, unsigned flags, void* stream,
                         const void* next, size_t next_bytes) {
    if (next && !aligned(next, 16))
        return fail(W4A8_ERR_ALIGN, "w4a8_linear_prefetch: next needs 16-byte alignment");
    PrefetchScope scope(next, next_bytes);
    return w4a8_linear(X, M, K, Wq, sw, N, Y, nullptr, nullptr, nullptr, ws, ws_bytes, flags, stream);
}

int w4a8_linear_grouped_prefetch(const uint16_t* X, int64_t M, int64_t K, int G, const uint8_t* const* Wq,
                                 const float* const* sw, const int64_t* N, float* const* Y, void* ws,
                                 size_t ws_bytes, unsigned flags, void* stream, const void* next,
                                 size_t next_bytes) {
    if (next && !aligned(next, 16))
        return fail(W4A8_ERR_ALIGN, "w4a8_linear_grouped_prefetch: next needs 16-byte alignment");
    PrefetchScope scope(next, next_bytes);
    return w4a8_linear_grouped(X, M, K, G, Wq, sw, N, Y, ws, ws_bytes, flags, stream);
}

}  // extern "C"

// C ABI of the library (declared in include/fa.h): argument validation, TMA
// tensor-map construction, kernel dispatch and error reporting.  No device
// memory is allocated here; every buffer, including scratch, is the caller's.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <climits>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "common.cuh"

namespace {

__device__ unsigned int g_fa_error_word;

thread_local char t_last_error[512] = "";

fa_status fail(fa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int cc_major = 0;
    unsigned int* err_word = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device facts, looked up once per device with that device current.
fa_status device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        d.sms = prop.multiProcessorCount;
        d.cc_major = prop.major;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fa_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        d.err_word = reinterpret_cast<unsigned int*>(p);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    if (d.cc_major != 10) return fail(FA_ERR_UNSUPPORTED, "needs a compute capability 10.x (Blackwell) device");
    *out = &d;
    return FA_OK;
}

// 3-D view [BH][N][d] of a contiguous [B,H,N,d] tensor, box {box_inner, box_rows, 1}.
fa_status make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, int d, int N, int BH,
                      int box_inner, int box_rows, CUtensorMapSwizzle sw) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * elem_bytes, (cuuint64_t)N * d * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FA_OK;
}

// Token-major packed tensor [total, heads, d] (bf16): TMA dims (d, head, token),
// boxes of 64 head-dim values x 1 head x box_rows consecutive tokens -- in
// shared memory the same [box_rows][128 bytes] tile as the [B,H,N,d] maps give.
fa_status make_map_tok(CUtensorMap* m, const void* base, int d, int heads, int total, int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (packed) failed (%d)", (int)r);
    return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_common(int B, int H, int N, int d, float scale) {
    if (B <= 0 || H <= 0 || N <= 0) return fail(FA_ERR_INVALID_ARG, "B, H, N must be positive (got %d, %d, %d)", B, H, N);
    if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
    if ((long long)B * H > (1ll << 30) || (long long)B * H * N * d > (1ll << 40))
        return fail(FA_ERR_INVALID_ARG, "problem too large");
    return FA_OK;
}

#define FA_CHECK_PTR(p)                                                                         \
    do {                                                                                        \
        if (!(p)) return fail(FA_ERR_INVALID_ARG, "%s must not be NULL", #p);                   \
        if (!aligned16(p)) return fail(FA_ERR_INVALID_ARG, "%s must be 16-byte aligned", #p); \
    } while (0)

#define FA_TRY(x)                           \
    do {                                    \
        fa_status _s = (x);                 \
        if (_s != FA_OK) return _s;         \
    } while (0)

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int grid_for_items(long items, int sms) { return (int)(items < sms ? items : sms); }

int bw_grid(const DeviceInfo* dev) { return dev->sms * 8; }

struct BwdLayout {
    size_t lse2, dvec, dqacc, q, k, v, dout, total;
};

BwdLayout bwd_layout(fa_dtype dt, int B, int H, int N, int d) {
    const size_t BH = (size_t)B * H, Np = round_up((size_t)N, 128);
    BwdLayout L;
    size_t off = 0;
    L.lse2 = off; off = round_up(off + BH * Np * 4, 256);
    L.dvec = off; off = round_up(off + BH * Np * 4, 256);
    L.dqacc = off; off = round_up(off + BH * Np * d * 4, 256);
    const size_t nb = BH * N * d * 2;
    if (dt == FA_F32) {
        L.q = off; off = round_up(off + nb, 256);
        L.k = off; off = round_up(off + nb, 256);
        L.v = off; off = round_up(off + nb, 256);
        L.dout = off; off = round_up(off + nb, 256);
    } else {
        L.q = L.k = L.v = L.dout = 0;
    }
    L.total = off;
    return L;
}

// Backward scratch (statistics, dQ accumulator; float32 inputs: their bf16
// copies), 0 for an unsupported shape.
size_t bwd_ws_bytes(fa_dtype dtype, int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    return bwd_layout(dtype, B, H, N, d).total;
}

// SM count of the current device, or the GB300's 152 when no device is
// visible (so that the split plan can be inspected on a host without a GPU).
int sm_count_or_default() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();
        return fa::kNumSMsDefault;
    }
    return sms;
}

// Split-key plan of a forward call.  Work is counted in key blocks of 128 with
// a fixed cost of two blocks per work unit (prologue, epilogue).  Automatic
// (requested = 0): whole items fill r full rounds of `sms` units and the
// remaining items are cut into s in [2, 4] key ranges, choosing (r, s) with the
// least estimated time (ties: more whole items, fewer ranges); kept only if it
// beats the unsplit schedule by more than 5%.  Causal items (unequal lengths,
// already balanced by the snake order) and key-padded batches are not split
// automatically.  requested = 1: no split; >= 2: every item in that many
// ranges (at most 64), the FlashDecoding form for few heads and long keys.
struct SplitPlan {
    int num_whole = 0, splits = 1;
    long long partials = 0;
    size_t o_bytes = 0, bytes = 0;
};
SplitPlan plan_split(int B, int H, int N, int d, bool causal, bool has_kv, int requested, int sms) {
    SplitPlan P;
    const long long items = (long long)B * H * ((N + 255) / 256);
    const int nb = (N + 127) / 128;
    long long whole = items;
    int S = 1;
    if (requested >= 2) {
        S = requested < 64 ? requested : 64;
        whole = 0;
    } else if (requested == 0 && !causal && !has_kv && nb >= 2) {
        const double unit = nb + 2.0;
        const double base = (double)((items + sms - 1) / sms) * unit;
        double best = base;
        for (long long r = items / sms; r >= 0; --r) {
            for (int s = 2; s <= 4 && s <= nb; ++s) {
                const long long tail = items - r * sms;
                const double t = (double)r * unit + (double)((tail * s + sms - 1) / sms) * ((double)nb / s + 2.0);
                if (t < best - 1e-9) {
                    best = t;
                    S = s;
                    whole = r * sms;
                }
            }
        }
        if (best > 0.95 * base) {
            S = 1;
            whole = items;
        }
    }
    P.num_whole = (int)whole;
    if (S > 1) {
        P.splits = S;
        P.partials = (items - whole) * S;
        P.o_bytes = round_up((size_t)P.partials * 256 * d * 4, 256);
        P.bytes = P.o_bytes + round_up((size_t)P.partials * 256 * 4, 256);
    }
    return P;
}

// Split plan of rectangular attention (Nq query rows, Nk keys).  Decode shapes
// have few items (B * H * ceil(Nq / 256)) of similar length whatever the
// masks, so when they fill less than half the GPU every item is cut into
// enough key ranges for ~2 x SMs units (at most one per key block, at most
// 64); with more items nothing is split unless num_splits asks for it.
SplitPlan plan_split_rect(int B, int H, int Nq, int Nk, int d, int requested, int sms) {
    const long long items = (long long)B * H * ((Nq + 255) / 256);
    const int nb = (Nk + 127) / 128;
    SplitPlan P;
    int S = 1;
    long long whole = items;
    if (requested >= 2) {
        S = requested < 64 ? requested : 64;
        whole = 0;
    } else if (requested == 0 && items * 2 <= sms && nb >= 2) {
        S = (int)((2LL * sms + items - 1) / items);
        S = S < nb ? S : nb;
        S = S < 64 ? S : 64;
        whole = 0;
    }
    P.num_whole = (int)whole;
    if (S > 1) {
        P.splits = S;
        P.partials = (items - whole) * S;
        P.o_bytes = round_up((size_t)P.partials * 256 * d * 4, 256);
        P.bytes = P.o_bytes + round_up((size_t)P.partials * 256 * 4, 256);
    }
    return P;
}

fa_status fwd_impl(fa_dtype dtype, int block_c, bool fp8, const void* q, const void* k, const void* v, const float* sq,
                   const float* sk, const float* sv, void* o, float* lse, int B, int H, int N, int d, float scale,
                   int causal, const int* kv_lens, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                   int num_splits = 1, void* split_ws = nullptr, size_t split_ws_bytes = 0, int Hkv = 0,
                   int win_left = -1, int win_right = -1, const int* row_ptr = nullptr,
                   const int* col_idx = nullptr) {
    FA_TRY(check_common(B, H, N, d, scale));
    const bool sparse = row_ptr != nullptr;
    if (sparse && (dtype != FA_BF16 || fp8)) return fail(FA_ERR_UNSUPPORTED, "block-sparse attention needs bf16 inputs");
    if (sparse && !col_idx) return fail(FA_ERR_INVALID_ARG, "col_idx must not be NULL");
    if (sparse && (win_left >= 0 || win_right >= 0))
        return fail(FA_ERR_UNSUPPORTED, "block lists and a sliding window cannot be combined");
    if (win_left < -1 || win_right < -1) return fail(FA_ERR_INVALID_ARG, "window edges must be >= -1");
    const bool window = win_left >= 0 || win_right >= 0;
    if (window && (dtype != FA_BF16 || fp8)) return fail(FA_ERR_UNSUPPORTED, "the sliding window needs bf16 inputs");
    if (window && block_c == 64) return fail(FA_ERR_UNSUPPORTED, "the sliding window uses 128-key blocks");
    if (window && num_splits > 1) return fail(FA_ERR_UNSUPPORTED, "the sliding window is not split over keys");
    if (Hkv == 0) Hkv = H;
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    if (Hkv != H && dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "shared key/value heads need bf16 inputs");
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    if (fp8) {
        if (d != 128) return fail(FA_ERR_UNSUPPORTED, "the FP8 forward needs d = 128");
        FA_CHECK_PTR(sq);
        FA_CHECK_PTR(sk);
        FA_CHECK_PTR(sv);
    }
    if (block_c != 0 && block_c != 64 && block_c != 128) return fail(FA_ERR_INVALID_ARG, "block_c must be 0, 64 or 128");
    if (fp8 && block_c == 64) return fail(FA_ERR_UNSUPPORTED, "the FP8 forward uses 128-key blocks");
    if (dtype != FA_BF16 && dtype != FA_F32) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    const int BH = B * H, BHkv = B * Hkv;
    const size_t n = (size_t)BH * N * d;
    const bool split = (dtype == FA_F32);
    const void *qb = q, *kb = k, *vb = v, *qlo = q, *klo = k;
    if (split) {
        // float32 inputs: q, k as bf16 hi + lo parts (scores from three bf16
        // products), v rounded to bf16
        const size_t part = round_up(n * 2, 256);
        if (workspace_bytes < 5 * part) return fail(FA_ERR_INVALID_ARG, "workspace too small");
        FA_CHECK_PTR(workspace);
        char* ws = reinterpret_cast<char*>(workspace);
        cudaError_t e;
        if ((e = fa::launch_f32_split_bf16((const float*)q, ws, ws + part, n, bw_grid(dev), stream)) != cudaSuccess)
            return cuda_fail(e, "float32 split launch");
        if ((e = fa::launch_f32_split_bf16((const float*)k, ws + 2 * part, ws + 3 * part, n, bw_grid(dev), stream)) !=
            cudaSuccess)
            return cuda_fail(e, "float32 split launch");
        if ((e = fa::launch_f32_to_bf16((const float*)v, ws + 4 * part, n, bw_grid(dev), stream)) != cudaSuccess)
            return cuda_fail(e, "float32 -> bf16 launch");
        qb = ws; qlo = ws + part; kb = ws + 2 * part; klo = ws + 3 * part; vb = ws + 4 * part;
        if (d == 128 && block_c == 128)
            return fail(FA_ERR_UNSUPPORTED, "float32 inputs with d = 128 use 64-key blocks");
        if (block_c == 0) block_c = (d == 128 || N <= 128) ? 64 : 128;
    }
    if (num_splits < 0) return fail(FA_ERR_INVALID_ARG, "num_splits must be >= 0");
    const SplitPlan P = (dtype == FA_BF16 && !window && !sparse)
                            ? plan_split(B, H, N, d, causal != 0, kv_lens != nullptr, num_splits, dev->sms)
                            : SplitPlan{};
    if (window || sparse) block_c = 128;
    if (P.splits > 1) block_c = 128;  // the split-key instances use 128-key blocks
    if (block_c == 0) block_c = (N <= 128 && !fp8) ? 64 : 128;
    fa::FwdMaps m;
    if (fp8) {
        FA_TRY(make_map_3d(&m.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qb, d, N, BH, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
        FA_TRY(make_map_3d(&m.k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kb, d, N, BHkv, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
        FA_TRY(make_map_3d(&m.v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, vb, d, N, BHkv, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
        m.q_lo = m.q;
        m.k_lo = m.k;
    } else {
        const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        FA_TRY(make_map_3d(&m.q, bf, 2, qb, d, N, BH, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
        FA_TRY(make_map_3d(&m.k, bf, 2, kb, d, N, BHkv, 64, block_c, CU_TENSOR_MAP_SWIZZLE_128B));
        FA_TRY(make_map_3d(&m.v, bf, 2, vb, d, N, BHkv, 64, block_c, CU_TENSOR_MAP_SWIZZLE_128B));
        FA_TRY(make_map_3d(&m.q_lo, bf, 2, qlo, d, N, BH, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
        FA_TRY(make_map_3d(&m.k_lo, bf, 2, klo, d, N, BHkv, 64, block_c, CU_TENSOR_MAP_SWIZZLE_128B));
    }
    fa::FwdParams p;
    memset(&p, 0, sizeof(p));
    p.B = B; p.H = H; p.N = N; p.Hkv = Hkv;
    p.num_qp = (N + 255) / 256;
    p.num_items = BH * p.num_qp;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kv_lens = kv_lens;
    p.o = o;
    p.lse = lse;
    p.sq = sq; p.sk = sk; p.sv = sv;
    p.nblk = (N + 63) / 64;
    p.err = dev->err_word;
    p.num_whole = (P.splits > 1) ? P.num_whole : p.num_items;
    p.splits = P.splits;
    p.num_units = p.num_whole + (int)P.partials;
    if (P.splits > 1) {
        if (!split_ws || split_ws_bytes < P.bytes)
            return fail(FA_ERR_INVALID_ARG, "split workspace too small (%zu bytes, need %zu)", split_ws_bytes, P.bytes);
        FA_CHECK_PTR(split_ws);
        p.o_part = reinterpret_cast<float*>(split_ws);
        p.lse_part = reinterpret_cast<float*>(reinterpret_cast<char*>(split_ws) + P.o_bytes);
    }
    const int grid = grid_for_items(p.num_units, dev->sms);
    cudaError_t e;
    if (sparse) {
        fa::FwdParamsSparse ps;
        memset(&ps, 0, sizeof(ps));
        static_cast<fa::FwdParams&>(ps) = p;
        ps.row_ptr = row_ptr;
        ps.col_idx = col_idx;
        ps.nqb = (N + 127) / 128;
        ps.nkb = (N + 127) / 128;
        e = fa::launch_fwd_sparse(d, causal != 0, m, ps, grid, stream);
    } else if (window) {
        // causal = the window's right edge at 0
        fa::FwdParamsWin pw;
        memset(&pw, 0, sizeof(pw));
        static_cast<fa::FwdParams&>(pw) = p;
        pw.win_left = win_left;
        pw.win_right = causal ? 0 : win_right;
        e = fa::launch_fwd_window(d, m, pw, grid, stream);
    } else if (P.splits > 1)
        e = fa::launch_fwd_splitk(d, fp8, causal != 0, m, p, grid, stream);
    else if (fp8)
        e = fa::launch_fwd_fp8_d128(causal != 0, m, p, grid, stream);
    else if (d == 128)
        e = fa::launch_fwd_bf16_d128(block_c, causal != 0, dtype == FA_F32, split, m, p, grid, stream);
    else
        e = fa::launch_fwd_bf16_d64(block_c, causal != 0, dtype == FA_F32, split, m, p, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    if (P.splits > 1) {
        e = fa::launch_lse_merge(p.o_part, p.lse_part, P.num_whole, p.num_items - P.num_whole, P.splits, causal != 0, BH,
                                 p.num_qp, N, d, o, lse, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split merge launch");
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_version(void) { return (0 << 16) | 1; }

const char* fa_last_error(void) { return t_last_error; }

fa_status fa_check_device_status(fa_stream_t stream) {
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int word = 0;
    e = cudaMemcpy(&word, dev->err_word, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word) {
        const unsigned int zero = 0;
        e = cudaMemcpy(dev->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        if (word & fa::kErrCheckMask)
            return fail(FA_ERR_CHECK, "a device access check of the checked build failed (error bits 0x%x)", word);
        return fail(FA_ERR_TIMEOUT, "a kernel pipeline wait timed out (error bits 0x%x)", word);
    }
    return FA_OK;
}

fa_status fa_selftest_quantiser_division(const float* x, const float* s, int ns, size_t n, float* q_fast,
                                        float* q_ieee, fa_stream_t stream) {
    if (!x || !s || !q_fast || !q_ieee) return fail(FA_ERR_INVALID_ARG, "null pointer");
    if (ns <= 0) return fail(FA_ERR_INVALID_ARG, "ns must be positive");
    cudaError_t e = fa::launch_shared_div_check(x, s, ns, n, q_fast, q_ieee, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "division self-test launch");
    return FA_OK;
}

fa_status fa_selftest_wait_timeout(unsigned int limit_us, int* waited_out, fa_stream_t stream) {
    FA_CHECK_PTR(waited_out);
    if (limit_us == 0 || limit_us > 1000000u) return fail(FA_ERR_INVALID_ARG, "limit_us must be in [1, 1e6]");
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    cudaError_t e = fa::launch_wait_selftest(dev->err_word, limit_us, waited_out, stream);
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return FA_OK;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, const int* kv_lens, fa_stream_t stream) {
    return fwd_impl(FA_BF16, 0, false, q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, N, d, scale, causal, kv_lens,
                    nullptr, 0, stream);
}

size_t fa_fwd_split_workspace_size(int B, int H, int N, int d, int causal, int has_kv_lens, int num_splits) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || num_splits < 0) return 0;
    return plan_split(B, H, N, d, causal != 0, has_kv_lens != 0, num_splits, sm_count_or_default()).bytes;
}

int fa_fwd_split_count(int B, int H, int N, int d, int causal, int has_kv_lens, int num_splits) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || num_splits < 0) return 1;
    return plan_split(B, H, N, d, causal != 0, has_kv_lens != 0, num_splits, sm_count_or_default()).splits;
}

fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                       float scale, int causal, const int* kv_lens, int num_splits, void* workspace,
                       size_t workspace_bytes, fa_stream_t stream) {
    return fwd_impl(FA_BF16, 0, false, q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, N, d, scale, causal, kv_lens,
                    nullptr, 0, stream, num_splits, workspace, workspace_bytes);
}

// The rectangular forward packs the query rows of each key/value head's
// group (contiguous in [B, H, Nq, d]): B * Hkv "heads" of (H / Hkv) * Nq rows.
size_t fa_fwd_rect_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || Hkv < 1 || H % Hkv != 0 || (d != 64 && d != 128) ||
        num_splits < 0)
        return 0;
    return plan_split_rect(B, Hkv, (H / Hkv) * Nq, Nk, d, num_splits, sm_count_or_default()).bytes;
}

int fa_fwd_rect_split_count(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || Hkv < 1 || H % Hkv != 0 || (d != 64 && d != 128) ||
        num_splits < 0)
        return 1;
    return plan_split_rect(B, Hkv, (H / Hkv) * Nq, Nk, d, num_splits, sm_count_or_default()).splits;
}

fa_status fa_fwd_rect(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Nq,
                      int Nk, int d, float scale, int causal, const int* kv_lens, int num_splits, void* workspace,
                      size_t workspace_bytes, fa_stream_t stream) {
    FA_TRY(check_common(B, H, Nq, d, scale));
    if (Nk <= 0) return fail(FA_ERR_INVALID_ARG, "Nk must be positive");
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    if (num_splits < 0) return fail(FA_ERR_INVALID_ARG, "num_splits must be >= 0");
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    const int R = (H / Hkv) * Nq;  // packed query rows per key/value head
    if ((long long)(H / Hkv) * Nq > (1LL << 30)) return fail(FA_ERR_INVALID_ARG, "too many query rows");
    const SplitPlan P = plan_split_rect(B, Hkv, R, Nk, d, num_splits, dev->sms);
    const int BHkv = B * Hkv;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    fa::FwdMaps m;
    FA_TRY(make_map_3d(&m.q, bf, 2, q, d, R, BHkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&m.k, bf, 2, k, d, Nk, BHkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&m.v, bf, 2, v, d, Nk, BHkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    m.q_lo = m.q;
    m.k_lo = m.k;
    fa::FwdParamsRect p;
    memset(&p, 0, sizeof(p));
    p.B = B; p.H = Hkv; p.N = R; p.Hkv = Hkv;
    p.num_qp = (R + 255) / 256;
    p.num_items = BHkv * p.num_qp;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kv_lens = kv_lens;
    p.o = o;
    p.lse = lse;
    p.err = dev->err_word;
    p.num_whole = (P.splits > 1) ? P.num_whole : p.num_items;
    p.splits = P.splits;
    p.num_units = p.num_whole + (int)P.partials;
    p.Nk = Nk;
    p.coff = Nk - Nq;
    p.qmod = Nq;
    if (P.splits > 1) {
        if (!workspace || workspace_bytes < P.bytes)
            return fail(FA_ERR_INVALID_ARG, "split workspace too small (%zu bytes, need %zu)", workspace_bytes, P.bytes);
        p.o_part = reinterpret_cast<float*>(workspace);
        p.lse_part = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + P.o_bytes);
    }
    cudaError_t e = fa::launch_fwd_rect(d, causal != 0, m, p, grid_for_items(p.num_units, dev->sms), stream);
    if (e != cudaSuccess) return cuda_fail(e, "rectangular forward launch");
    if (P.splits > 1) {
        e = fa::launch_lse_merge(p.o_part, p.lse_part, P.num_whole, p.num_items - P.num_whole, P.splits, causal != 0,
                                 BHkv, p.num_qp, R, d, o, lse, stream);
        if (e != cudaSuccess) return cuda_fail(e, "split merge launch");
    }
    return FA_OK;
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
                     int d, float scale, int causal, const int* kv_lens, fa_stream_t stream) {
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    return fwd_impl(FA_BF16, 0, false, q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, N, d, scale, causal, kv_lens,
                    nullptr, 0, stream, 1, nullptr, 0, Hkv);
}

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                        int N, int d, float scale, int causal, int window_left, int window_right,
                        const int* kv_lens, fa_stream_t stream) {
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    return fwd_impl(FA_BF16, 0, false, q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, N, d, scale, causal, kv_lens,
                    nullptr, 0, stream, 1, nullptr, 0, Hkv, window_left, window_right);
}

fa_status fa_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int Hkv, int N, int d, float scale, int causal, const int* row_ptr,
                              const int* col_idx, const int* kv_lens, fa_stream_t stream) {
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    if (!row_ptr || !col_idx) return fail(FA_ERR_INVALID_ARG, "row_ptr and col_idx must not be NULL");
    return fwd_impl(FA_BF16, 0, false, q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, N, d, scale, causal, kv_lens,
                    nullptr, 0, stream, 1, nullptr, 0, Hkv, -1, -1, row_ptr, col_idx);
}

}  // extern "C"

namespace {

// Token-major forward ([total, H, d] tensors): packed sequences from
// cu_seqlens, or, with cu_seqlens NULL, batch sequences of max_seqlen tokens
// each (the [B, N, H, d] layout, LSE [B, H, N]).
fa_status fwd_packed_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                          int batch, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                          fa_stream_t stream, const int* cu_seqlens_k = nullptr, int total_k = -1,
                          int win_left = -1, int win_right = -1) {
    if (total_k < 0) total_k = total;
    if (win_left < -1 || win_right < -1) return fail(FA_ERR_INVALID_ARG, "window edges must be >= -1");
    const bool window = win_left >= 0 || win_right >= 0;
    if (window && cu_seqlens_k) return fail(FA_ERR_UNSUPPORTED, "the sliding window needs one range per sequence");
    if (total_k <= 0) return fail(FA_ERR_INVALID_ARG, "total_k must be positive");
    FA_TRY(check_common(batch, H, max_seqlen, d, scale));
    if (total <= 0) return fail(FA_ERR_INVALID_ARG, "total must be positive");
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    fa::FwdMaps m;
    FA_TRY(make_map_tok(&m.q, q, d, H, total, 128));
    FA_TRY(make_map_tok(&m.k, k, d, Hkv, total_k, 128));
    FA_TRY(make_map_tok(&m.v, v, d, Hkv, total_k, 128));
    m.q_lo = m.q;
    m.k_lo = m.k;
    fa::FwdParams p;
    memset(&p, 0, sizeof(p));
    p.B = batch; p.H = H; p.N = max_seqlen; p.Hkv = Hkv;
    p.num_qp = (max_seqlen + 255) / 256;
    p.num_items = batch * H * p.num_qp;
    p.num_units = p.num_whole = p.num_items;
    p.splits = 1;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.o = o;
    p.lse = lse;
    p.cu_seqlens = cu_seqlens;
    p.cu_seqlens_k = cu_seqlens_k;
    p.total = total;
    p.err = dev->err_word;
    cudaError_t e;
    if (window) {  // causal = the window's right edge at 0
        fa::FwdParamsWin pw;
        memset(&pw, 0, sizeof(pw));
        static_cast<fa::FwdParams&>(pw) = p;
        pw.win_left = win_left;
        pw.win_right = causal ? 0 : win_right;
        e = fa::launch_fwd_varlen_window(d, m, pw, grid_for_items(p.num_items, dev->sms), stream);
    } else {
        e = fa::launch_fwd_varlen(d, causal != 0, m, p, grid_for_items(p.num_items, dev->sms), stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "varlen forward launch");
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                        int batch, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                        fa_stream_t stream) {
    if (!cu_seqlens) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    return fwd_packed_impl(q, k, v, o, lse, cu_seqlens, batch, total, max_seqlen, H, Hkv, d, scale, causal, stream);
}

fa_status fa_fwd_varlen_window(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                               int batch, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                               int window_left, int window_right, fa_stream_t stream) {
    if (!cu_seqlens) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    return fwd_packed_impl(q, k, v, o, lse, cu_seqlens, batch, total, max_seqlen, H, Hkv, d, scale, causal, stream,
                           nullptr, -1, window_left, window_right);
}

fa_status fa_fwd_varlen_kv(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                           const int* cu_seqlens_k, int batch, int total_q, int total_k, int max_seqlen_q, int H,
                           int Hkv, int d, float scale, int causal, fa_stream_t stream) {
    if (!cu_seqlens_q || !cu_seqlens_k) return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must not be NULL");
    return fwd_packed_impl(q, k, v, o, lse, cu_seqlens_q, batch, total_q, max_seqlen_q, H, Hkv, d, scale, causal,
                           stream, cu_seqlens_k, total_k);
}

fa_status fa_fwd_bnhd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int N, int H, int Hkv,
                      int d, float scale, int causal, fa_stream_t stream) {
    if ((long long)B * N > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B * N exceeds the 32-bit token index");
    return fwd_packed_impl(q, k, v, o, lse, nullptr, B, B * N, N, H, Hkv, d, scale, causal, stream);
}

size_t fa_fwd_workspace_size(fa_dtype dtype, int B, int H, int N, int d) {
    if (dtype != FA_F32 || B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
    return 5 * round_up((size_t)B * H * N * d * 2, 256);
}

fa_status fa_fwd_ex(fa_dtype dtype, int block_c, const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int N, int d, float scale, int causal, const int* kv_lens, void* workspace,
                    size_t workspace_bytes, fa_stream_t stream) {
    return fwd_impl(dtype, block_c, false, q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, N, d, scale, causal,
                    kv_lens, workspace, workspace_bytes, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) { return bwd_ws_bytes(FA_BF16, B, H, N, d); }

}  // extern "C"

namespace {

struct BwdCtx {
    DeviceInfo* dev;
    BwdLayout L;
    int BH, Np;
    char* ws;
};

fa_status bwd_setup(fa_dtype dtype, int B, int H, int N, int d, float scale, void* workspace, size_t workspace_bytes,
                    BwdCtx* c) {
    FA_TRY(check_common(B, H, N, d, scale));
    FA_CHECK_PTR(workspace);
    if (dtype != FA_BF16 && dtype != FA_F32) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    c->L = bwd_layout(dtype, B, H, N, d);
    if (workspace_bytes < c->L.total)
        return fail(FA_ERR_INVALID_ARG, "workspace too small (%zu < %zu bytes)", workspace_bytes, c->L.total);
    FA_TRY(device_info(&c->dev));
    c->BH = B * H;
    c->Np = (int)round_up((size_t)N, 128);
    c->ws = reinterpret_cast<char*>(workspace);
    return FA_OK;
}

fa_status bwd_pre_impl(const BwdCtx& c, bool f32, const void* o, const float* lse, const void* dout, int N, int d,
                       cudaStream_t stream) {
    cudaError_t e = fa::launch_bwd_pre(o, dout, f32, lse, reinterpret_cast<float*>(c.ws + c.L.lse2),
                                       reinterpret_cast<float*>(c.ws + c.L.dvec),
                                       reinterpret_cast<float*>(c.ws + c.L.dqacc), c.BH, N, c.Np, d, bw_grid(c.dev),
                                       stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
    return FA_OK;
}

// The float32 dQ accumulator [rows][d] as the target of the drain warps' tensor
// reductions: d = 128: [64 queries][32 head-dim] boxes, plain; d = 64:
// [32 queries][32 head-dim] boxes in the 128-byte swizzle they are staged in.
fa_status make_map_dqacc(CUtensorMap* m, float* dqacc, int d, long long rows, int box_rows = 0) {
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)(box_rows ? box_rows : (d == 128 ? 64 : 32))};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, dqacc, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, d == 128 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (dQ accumulator) failed (%d)", (int)r);
    return FA_OK;
}

// Units per key block for the grouped backward: the smallest divisor g of the
// group with items * g >= 2 * SMs (1 when the key blocks already fill the GPU
// twice over), so that the longest unit is short next to a CTA's share.
int choose_gsplit(long items, int group, int sms) {
    if (items >= 2L * sms || group < 2) return 1;
    for (int g = 2; g < group; ++g)
        if (group % g == 0 && items * g >= 2L * sms) return g;
    return group;
}

// Deterministic backward: the number of dQ accumulators, from the shape
// alone (so that the result does not depend on the device): enough that the
// key blocks of one key/value head in one round of a 152-SM grid, which run
// at the same time in key-block-major order, land in different accumulators;
// at most 8 and at most the number of key blocks.
constexpr int kDetMaxAcc = 8;  // the conversion kernel reads at most 8
int det_num_acc(int B, int Hkv, int N) {
    const long heads = (long)B * Hkv, kt = (N + 127) / 128;
    long a = (fa::kNumSMsDefault + heads - 1) / heads + 1;
    if (a > kDetMaxAcc) a = kDetMaxAcc;
    if (a > kt) a = kt;
    return (int)(a < 1 ? 1 : a);
}
// Turn counters: 4 per dQ tile of BR rows, per accumulator.
size_t det_turn_bytes(int nacc, int B, int H, int N, int d) {
    const size_t Np = round_up((size_t)N, 128);
    return (size_t)nacc * B * H * (Np / (d == 128 ? 64 : 128)) * 4 * sizeof(int);
}
size_t det_acc_bytes(int B, int H, int N, int d) { return (size_t)B * H * round_up((size_t)N, 128) * d * sizeof(float); }

size_t dkv_part_bytes(int g, int B, int Hkv, int N, int d) { return (size_t)g * 2 * B * Hkv * N * d * sizeof(float); }

fa_status bwd_main_impl(const BwdCtx& c, bool f32, const void* qb, const void* kb, const void* vb, const void* gb,
                        void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                        cudaStream_t stream, int Hkv = 0, int win_left = -1, int win_right = -1,
                        const int* col_ptr = nullptr, const int* row_idx = nullptr, float* dkv_part = nullptr,
                        size_t part_bytes = 0, int Nk = -1, int* dq_turn = nullptr, int nacc = 1,
                        const int* row_ptr = nullptr, const int* col_idx = nullptr) {
    const int BH = c.BH, Np = c.Np;
    const bool rect = Nk >= 0;  // rectangular: N query rows, Nk keys
    if (!rect) Nk = N;
    if (Hkv == 0) Hkv = H;
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    const int BHkv = B * Hkv;
    float* dqacc = reinterpret_cast<float*>(c.ws + c.L.dqacc);
    const int BR = (d == 128) ? 64 : 128;
    CUtensorMap tq, tk, tv, tdo, tdq;
    FA_TRY(make_map_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, qb, d, N, BH, 64, BR, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tdo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, gb, d, N, BH, 64, BR, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kb, d, Nk, BHkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vb, d, Nk, BHkv, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    if ((long long)BH * Np * nacc >= (1LL << 31))
        return fail(FA_ERR_UNSUPPORTED, "dQ accumulator rows exceed the 32-bit tensor coordinate range");
    FA_TRY(make_map_dqacc(&tdq, dqacc, d, (long long)BH * Np * nacc));
    fa::BwdParams p;
    memset(&p, 0, sizeof(p));
    p.B = B; p.H = H; p.N = N; p.Np = Np; p.Hkv = Hkv;
    p.num_kt = (Nk + 127) / 128;
    p.num_items = BHkv * p.num_kt;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kv_lens = kv_lens;
    p.lse2 = reinterpret_cast<float*>(c.ws + c.L.lse2);
    p.dvec = reinterpret_cast<float*>(c.ws + c.L.dvec);
    p.dq_acc = dqacc;
    p.dk = dk;
    p.dv = dv;
    p.err = c.dev->err_word;
    // the grouped instances (shared heads, window, block lists) may split a
    // key block's query heads over several units when key blocks are few
    const bool grouped = Hkv != H || col_ptr || win_left >= 0 || win_right >= 0 || rect;
    p.gsplit = 1;
    if (grouped && dkv_part) {
        const int g = choose_gsplit(p.num_items, H / Hkv, c.dev->sms);
        if (g > 1 && part_bytes >= dkv_part_bytes(g, B, Hkv, Nk, d)) {
            p.gsplit = g;
            p.dkv_part = dkv_part;
            p.num_items *= g;
        }
    }
    const int grid = grid_for_items(p.num_items, c.dev->sms);
    cudaError_t e;
    if (dq_turn) {
        // deterministic: zeroed turn counters, one per quarter of a dQ tile
        auto set_det = [&](auto& pd) {
            pd.nqt = Np / BR;
            pd.dq_turn = dq_turn;
            pd.nacc = nacc;
        };
        e = cudaMemsetAsync(dq_turn, 0, det_turn_bytes(nacc, B, H, N, d), stream);
        if (e == cudaSuccess) {
            if (rect) {
                fa::BwdDet<fa::BwdParamsRect> pd;
                memset(&pd, 0, sizeof(pd));
                static_cast<fa::BwdParams&>(pd) = p;
                pd.Nk = Nk;
                pd.coff = Nk - N;
                set_det(pd);
                e = fa::launch_bwd_main_det_rect(d, causal != 0, tq, tk, tv, tdo, tdq, pd, grid, stream);
            } else if (col_ptr) {
                fa::BwdDet<fa::BwdParamsSparse> pd;
                memset(&pd, 0, sizeof(pd));
                static_cast<fa::BwdParams&>(pd) = p;
                pd.col_ptr = col_ptr;
                pd.row_idx = row_idx;
                pd.nqb = (N + 127) / 128;
                pd.nkb = (N + 127) / 128;
                pd.row_ptr = row_ptr;
                pd.col_idx = col_idx;
                set_det(pd);
                e = fa::launch_bwd_main_det_sparse(d, causal != 0, tq, tk, tv, tdo, tdq, pd, grid, stream);
            } else if (win_left >= 0 || win_right >= 0) {
                fa::BwdDet<fa::BwdParamsWin> pd;
                memset(&pd, 0, sizeof(pd));
                static_cast<fa::BwdParams&>(pd) = p;
                pd.win_left = win_left;
                pd.win_right = causal ? 0 : win_right;
                set_det(pd);
                e = fa::launch_bwd_main_det_window(d, tq, tk, tv, tdo, tdq, pd, grid, stream);
            } else {
                fa::BwdParamsDet pd;
                memset(&pd, 0, sizeof(pd));
                static_cast<fa::BwdParams&>(pd) = p;
                set_det(pd);
                e = fa::launch_bwd_main_det(d, causal != 0, tq, tk, tv, tdo, tdq, pd, grid, stream);
            }
        }
    } else if (rect) {
        fa::BwdParamsRect pr;
        memset(&pr, 0, sizeof(pr));
        static_cast<fa::BwdParams&>(pr) = p;
        pr.Nk = Nk;
        pr.coff = Nk - N;
        e = fa::launch_bwd_main_rect(d, causal != 0, tq, tk, tv, tdo, tdq, pr, grid, stream);
    } else if (col_ptr) {
        fa::BwdParamsSparse ps;
        memset(&ps, 0, sizeof(ps));
        static_cast<fa::BwdParams&>(ps) = p;
        ps.col_ptr = col_ptr;
        ps.row_idx = row_idx;
        ps.nqb = (N + 127) / 128;
        ps.nkb = (N + 127) / 128;
        e = fa::launch_bwd_main_sparse(d, causal != 0, tq, tk, tv, tdo, tdq, ps, grid, stream);
    } else if (win_left >= 0 || win_right >= 0) {
        // causal = the window's right edge at 0
        fa::BwdParamsWin pw;
        memset(&pw, 0, sizeof(pw));
        static_cast<fa::BwdParams&>(pw) = p;
        pw.win_left = win_left;
        pw.win_right = causal ? 0 : win_right;
        e = fa::launch_bwd_main_window(d, tq, tk, tv, tdo, tdq, pw, grid, stream);
    } else {
        e = (Hkv != H) ? fa::launch_bwd_main_gqa(d, causal != 0, tq, tk, tv, tdo, tdq, p, grid, stream)
                       : fa::launch_bwd_main(d, causal != 0, f32, tq, tk, tv, tdo, tdq, p, grid, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "backward main launch");
    if (p.gsplit > 1) {
        e = fa::launch_dkv_sum(dkv_part, p.gsplit, (size_t)B * Hkv * Nk * d, dk, dv, bw_grid(c.dev), stream);
        if (e != cudaSuccess) return cuda_fail(e, "dK / dV partial sum launch");
    }
    return FA_OK;
}

fa_status bwd_dq_impl(const BwdCtx& c, bool f32, void* dq, int N, int d, float scale, cudaStream_t stream) {
    cudaError_t e = fa::launch_bwd_dq(reinterpret_cast<float*>(c.ws + c.L.dqacc), dq, f32, scale, c.BH, N, c.Np, d,
                                      c.dev->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "dQ conversion launch");
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H, int N, int d,
                            void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, 1.0f, workspace, workspace_bytes, &c));
    return bwd_pre_impl(c, false, o, lse, dout, N, d, stream);
}

fa_status fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv, int B, int H,
                      int N, int d, float scale, int causal, const int* kv_lens, void* workspace,
                      size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, scale, workspace, workspace_bytes, &c));
    return bwd_main_impl(c, false, q, k, v, dout, dk, dv, B, H, N, d, scale, causal, kv_lens, stream);
}

fa_status fa_bwd_dq(void* dq, int B, int H, int N, int d, float scale, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
    FA_CHECK_PTR(dq);
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, scale, workspace, workspace_bytes, &c));
    return bwd_dq_impl(c, false, dq, N, d, scale, stream);
}

fa_status fa_bwd_ex(fa_dtype dtype, const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                    const int* kv_lens, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    BwdCtx c{};
    FA_TRY(bwd_setup(dtype, B, H, N, d, scale, workspace, workspace_bytes, &c));
    const bool f32 = dtype == FA_F32;
    const void *qb = q, *kb = k, *vb = v, *gb = dout;
    if (f32) {
        const size_t n = (size_t)c.BH * N * d;
        const void* src[4] = {q, k, v, dout};
        const size_t dst[4] = {c.L.q, c.L.k, c.L.v, c.L.dout};
        for (int i = 0; i < 4; ++i) {
            cudaError_t e = fa::launch_f32_to_bf16((const float*)src[i], c.ws + dst[i], n, bw_grid(c.dev), stream);
            if (e != cudaSuccess) return cuda_fail(e, "float32 -> bf16 launch");
        }
        qb = c.ws + c.L.q; kb = c.ws + c.L.k; vb = c.ws + c.L.v; gb = c.ws + c.L.dout;
    }
    FA_TRY(bwd_pre_impl(c, f32, o, lse, dout, N, d, stream));
    FA_TRY(bwd_main_impl(c, f32, qb, kb, vb, gb, dk, dv, B, H, N, d, scale, causal, kv_lens, stream));
    return bwd_dq_impl(c, f32, dq, N, d, scale, stream);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, float scale, int causal,
                     const int* kv_lens, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, scale, workspace, workspace_bytes, &c));
    FA_TRY(bwd_pre_impl(c, false, o, lse, dout, N, d, stream));
    const size_t base = round_up(c.L.total, 256);
    float* part = workspace_bytes > base ? reinterpret_cast<float*>(c.ws + base) : nullptr;
    FA_TRY(bwd_main_impl(c, false, q, k, v, dout, dk, dv, B, H, N, d, scale, causal, kv_lens, stream, Hkv, -1, -1,
                         nullptr, nullptr, part, part ? workspace_bytes - base : 0));
    return bwd_dq_impl(c, false, dq, N, d, scale, stream);
}

// Block lists of 128 x 128 blocks: the transposed lists live after the
// backward's own workspace, 256-byte aligned.
constexpr int kMaxSparseBlocks = 12000;  // the transposition keeps nkb + 1 counters in shared memory

static size_t sparse_lists_bytes(int N) {
    const size_t nb = (size_t)(N + 127) / 128;
    return round_up((nb + 1 + nb * nb) * sizeof(int), 256);
}

size_t fa_bwd_block_sparse_workspace_size(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    return round_up(bwd_ws_bytes(FA_BF16, B, H, N, d), 256) + sparse_lists_bytes(N);
}

fa_status fa_bwd_block_sparse(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                              float scale, int causal, const int* row_ptr, const int* col_idx, const int* kv_lens,
                              void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    if (!row_ptr || !col_idx) return fail(FA_ERR_INVALID_ARG, "row_ptr and col_idx must not be NULL");
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    if (N > 0 && (N + 127) / 128 > kMaxSparseBlocks)
        return fail(FA_ERR_UNSUPPORTED, "block-sparse attention takes at most %d blocks", kMaxSparseBlocks);
    const size_t need = fa_bwd_block_sparse_workspace_size(B, H, N, d);
    if (workspace_bytes < need)
        return fail(FA_ERR_INVALID_ARG, "workspace too small (%zu < %zu bytes)", workspace_bytes, need);
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, scale, workspace, workspace_bytes, &c));
    const int nb = (N + 127) / 128;
    int* col_ptr = reinterpret_cast<int*>(c.ws + round_up(bwd_ws_bytes(FA_BF16, B, H, N, d), 256));
    int* row_idx = col_ptr + nb + 1;
    cudaError_t e = fa::launch_block_lists_transpose(row_ptr, col_idx, nb, nb, col_ptr, row_idx, stream);
    if (e != cudaSuccess) return cuda_fail(e, "block list transposition launch");
    FA_TRY(bwd_pre_impl(c, false, o, lse, dout, N, d, stream));
    FA_TRY(bwd_main_impl(c, false, q, k, v, dout, dk, dv, B, H, N, d, scale, causal, kv_lens, stream, Hkv, -1, -1,
                         col_ptr, row_idx));
    return bwd_dq_impl(c, false, dq, N, d, scale, stream);
}

size_t fa_bwd_rect_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || Hkv < 1 || H % Hkv != 0 || (d != 64 && d != 128)) return 0;
    const size_t base = round_up(bwd_ws_bytes(FA_BF16, B, H, Nq, d), 256);
    const int g = choose_gsplit((long)B * Hkv * ((Nk + 127) / 128), H / Hkv, sm_count_or_default());
    return g > 1 ? base + dkv_part_bytes(g, B, Hkv, Nk, d) : base;
}

fa_status fa_bwd_rect(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                      int causal, const int* kv_lens, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    if (Nk <= 0) return fail(FA_ERR_INVALID_ARG, "Nk must be positive");
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, Nq, d, scale, workspace, workspace_bytes, &c));
    FA_TRY(bwd_pre_impl(c, false, o, lse, dout, Nq, d, stream));
    const size_t base = round_up(c.L.total, 256);
    float* part = workspace_bytes > base ? reinterpret_cast<float*>(c.ws + base) : nullptr;
    FA_TRY(bwd_main_impl(c, false, q, k, v, dout, dk, dv, B, H, Nq, d, scale, causal, kv_lens, stream, Hkv, -1, -1,
                         nullptr, nullptr, part, part ? workspace_bytes - base : 0, Nk));
    return bwd_dq_impl(c, false, dq, Nq, d, scale, stream);
}

size_t fa_bwd_gqa_workspace_size(int B, int H, int Hkv, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || Hkv < 1 || H % Hkv != 0 || (d != 64 && d != 128)) return 0;
    const size_t base = round_up(bwd_ws_bytes(FA_BF16, B, H, N, d), 256);
    const int g = choose_gsplit((long)B * Hkv * ((N + 127) / 128), H / Hkv, sm_count_or_default());
    return g > 1 ? base + dkv_part_bytes(g, B, Hkv, N, d) : base;
}

fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                        float scale, int causal, int window_left, int window_right, const int* kv_lens,
                        void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    if (window_left < -1 || window_right < -1) return fail(FA_ERR_INVALID_ARG, "window edges must be >= -1");
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, scale, workspace, workspace_bytes, &c));
    FA_TRY(bwd_pre_impl(c, false, o, lse, dout, N, d, stream));
    const size_t base = round_up(c.L.total, 256);
    float* part = workspace_bytes > base ? reinterpret_cast<float*>(c.ws + base) : nullptr;
    FA_TRY(bwd_main_impl(c, false, q, k, v, dout, dk, dv, B, H, N, d, scale, causal, kv_lens, stream, Hkv, window_left,
                         window_right, nullptr, nullptr, part, part ? workspace_bytes - base : 0));
    return bwd_dq_impl(c, false, dq, N, d, scale, stream);
}

size_t fa_bwd_varlen_workspace_size(int batch, int max_seqlen, int H, int d) {
    if (batch <= 0 || max_seqlen <= 0 || H <= 0 || (d != 64 && d != 128)) return 0;
    const size_t R = (size_t)H * batch * round_up((size_t)max_seqlen, 128);
    return 2 * round_up(R * 4, 256) + round_up(R * d * 4, 256);
}

size_t fa_bwd_varlen_deterministic_workspace_size(int batch, int max_seqlen, int H, int Hkv, int d) {
    const size_t base = fa_bwd_varlen_workspace_size(batch, max_seqlen, H, d);
    if (base == 0 || Hkv < 1 || H % Hkv != 0) return 0;
    const int nacc = det_num_acc(batch, Hkv, max_seqlen);
    return base + (size_t)(nacc - 1) * det_acc_bytes(batch, H, max_seqlen, d) +
           det_turn_bytes(nacc, batch, H, max_seqlen, d);
}

size_t fa_bwd_bnhd_deterministic_workspace_size(int B, int N, int H, int Hkv, int d) {
    return fa_bwd_varlen_deterministic_workspace_size(B, N, H, Hkv, d);
}

}  // extern "C"

namespace {

// Token-major backward (see fwd_packed_impl; cu_seqlens NULL = uniform lengths).
fa_status bwd_packed_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens, int batch, int total,
                          int max_seqlen, int H, int Hkv, int d, float scale, int causal, void* workspace,
                          size_t workspace_bytes, fa_stream_t stream, bool det = false,
                          const int* cu_seqlens_k = nullptr, int total_k = -1, int max_seqlen_k = -1,
                          int win_left = -1, int win_right = -1) {
    if (total_k < 0) total_k = total;
    if (win_left < -1 || win_right < -1) return fail(FA_ERR_INVALID_ARG, "window edges must be >= -1");
    const bool window = win_left >= 0 || win_right >= 0;
    if (window && cu_seqlens_k) return fail(FA_ERR_UNSUPPORTED, "the packed sliding window takes one range per sequence");
    if (max_seqlen_k < 0) max_seqlen_k = max_seqlen;
    if (total_k <= 0 || max_seqlen_k <= 0) return fail(FA_ERR_INVALID_ARG, "total_k and max_seqlen_k must be positive");
    FA_TRY(check_common(batch, H, max_seqlen, d, scale));
    if (total <= 0) return fail(FA_ERR_INVALID_ARG, "total must be positive");
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    FA_CHECK_PTR(workspace);
    const size_t base = fa_bwd_varlen_workspace_size(batch, max_seqlen, H, d);
    const int nacc = det ? det_num_acc(batch, Hkv, max_seqlen_k) : 1;
    const size_t need = det ? base + (size_t)(nacc - 1) * det_acc_bytes(batch, H, max_seqlen, d) +
                                  det_turn_bytes(nacc, batch, H, max_seqlen, d)
                            : base;
    if (workspace_bytes < need) return fail(FA_ERR_INVALID_ARG, "workspace too small (%zu < %zu bytes)", workspace_bytes, need);
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    const int MSp = (int)round_up((size_t)max_seqlen, 128);
    const size_t R = (size_t)H * batch * MSp;
    char* ws = reinterpret_cast<char*>(workspace);
    float* lse2 = reinterpret_cast<float*>(ws);
    float* dvec = reinterpret_cast<float*>(ws + round_up(R * 4, 256));
    float* dqacc = reinterpret_cast<float*>(ws + 2 * round_up(R * 4, 256));
    cudaError_t e = fa::launch_bwd_pre_varlen(o, dout, lse, cu_seqlens, lse2, dvec, dqacc, H, batch, total, max_seqlen,
                                              MSp, d, bw_grid(dev), stream);
    if (e != cudaSuccess) return cuda_fail(e, "varlen preprocess launch");
    const int BR = (d == 128) ? 64 : 128;
    CUtensorMap tq, tk, tv, tdo, tdq;
    FA_TRY(make_map_tok(&tq, q, d, H, total, BR));
    FA_TRY(make_map_tok(&tdo, dout, d, H, total, BR));
    FA_TRY(make_map_tok(&tk, k, d, Hkv, total_k, 128));
    FA_TRY(make_map_tok(&tv, v, d, Hkv, total_k, 128));
    if ((long long)R * nacc >= (1LL << 31))
        return fail(FA_ERR_UNSUPPORTED, "dQ accumulator rows exceed the 32-bit tensor coordinate range");
    FA_TRY(make_map_dqacc(&tdq, dqacc, d, (long long)R * nacc));
    fa::BwdParams p;
    memset(&p, 0, sizeof(p));
    p.B = batch; p.H = H; p.N = max_seqlen; p.Np = MSp; p.Hkv = Hkv;
    p.num_kt = (max_seqlen_k + 127) / 128;
    p.num_items = batch * Hkv * p.num_kt;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq_acc = dqacc;
    p.dk = dk;
    p.dv = dv;
    p.cu_seqlens = cu_seqlens;
    p.cu_seqlens_k = cu_seqlens_k;
    p.total = total;
    p.err = dev->err_word;
    if (det) {
        // accumulators 1 .. nacc-1 follow the first (the last region), then the turn counters
        int* turn = reinterpret_cast<int*>(ws + base + (size_t)(nacc - 1) * R * d * sizeof(float));
        fa::BwdParamsDet pd;
        memset(&pd, 0, sizeof(pd));
        static_cast<fa::BwdParams&>(pd) = p;
        pd.nqt = MSp / (d == 128 ? 64 : 128);
        pd.dq_turn = turn;
        pd.nacc = nacc;
        e = cudaMemsetAsync(turn, 0, det_turn_bytes(nacc, batch, H, max_seqlen, d), stream);
        if (e == cudaSuccess && window) {  // causal = the window's right edge at 0
            fa::BwdDet<fa::BwdParamsWin> pw;
            memset(&pw, 0, sizeof(pw));
            static_cast<fa::BwdParams&>(pw) = p;
            pw.win_left = win_left;
            pw.win_right = causal ? 0 : win_right;
            pw.nqt = pd.nqt;
            pw.dq_turn = turn;
            pw.nacc = nacc;
            e = fa::launch_bwd_main_det_varlen_window(d, tq, tk, tv, tdo, tdq, pw, grid_for_items(p.num_items, dev->sms),
                                                      stream);
        } else if (e == cudaSuccess) {
            e = fa::launch_bwd_main_det_varlen(d, causal != 0, tq, tk, tv, tdo, tdq, pd,
                                               grid_for_items(p.num_items, dev->sms), stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "varlen deterministic backward launch");
        e = fa::launch_bwd_dq_det_varlen(dqacc, turn, cu_seqlens, dq, scale, H, batch, max_seqlen, MSp, d, nacc,
                                         bw_grid(dev), stream);
        if (e != cudaSuccess) return cuda_fail(e, "varlen dQ conversion launch");
        return FA_OK;
    }
    if (window) {  // causal = the window's right edge at 0
        fa::BwdParamsWin pw;
        memset(&pw, 0, sizeof(pw));
        static_cast<fa::BwdParams&>(pw) = p;
        pw.win_left = win_left;
        pw.win_right = causal ? 0 : win_right;
        e = fa::launch_bwd_main_varlen_window(d, tq, tk, tv, tdo, tdq, pw, grid_for_items(p.num_items, dev->sms),
                                              stream);
    } else {
        e = fa::launch_bwd_main_varlen(d, causal != 0, tq, tk, tv, tdo, tdq, p, grid_for_items(p.num_items, dev->sms),
                                       stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "varlen backward launch");
    e = fa::launch_bwd_dq_varlen(dqacc, cu_seqlens, dq, scale, H, batch, max_seqlen, MSp, d, bw_grid(dev), stream);
    if (e != cudaSuccess) return cuda_fail(e, "varlen dQ conversion launch");
    return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens, int batch, int total,
                        int max_seqlen, int H, int Hkv, int d, float scale, int causal, void* workspace,
                        size_t workspace_bytes, fa_stream_t stream) {
    if (!cu_seqlens) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    return bwd_packed_impl(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, batch, total, max_seqlen, H, Hkv, d, scale,
                           causal, workspace, workspace_bytes, stream);
}

size_t fa_bwd_bnhd_workspace_size(int B, int N, int H, int d) { return fa_bwd_varlen_workspace_size(B, N, H, d); }

fa_status fa_bwd_varlen_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens, int batch,
                               int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                               int window_left, int window_right, int deterministic, void* workspace,
                               size_t workspace_bytes, fa_stream_t stream) {
    if (!cu_seqlens) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    return bwd_packed_impl(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, batch, total, max_seqlen, H, Hkv, d, scale,
                           causal, workspace, workspace_bytes, stream, deterministic != 0, nullptr, -1, -1,
                           window_left, window_right);
}

size_t fa_bwd_varlen_kv_workspace_size(int batch, int max_seqlen_q, int max_seqlen_k, int H, int Hkv, int d,
                                       int deterministic) {
    const size_t base = fa_bwd_varlen_workspace_size(batch, max_seqlen_q, H, d);
    if (base == 0 || max_seqlen_k <= 0 || Hkv < 1 || H % Hkv != 0) return 0;
    if (!deterministic) return base;
    const int nacc = det_num_acc(batch, Hkv, max_seqlen_k);
    return base + (size_t)(nacc - 1) * det_acc_bytes(batch, H, max_seqlen_q, d) +
           det_turn_bytes(nacc, batch, H, max_seqlen_q, d);
}

fa_status fa_bwd_varlen_kv(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                           const int* cu_seqlens_k, int batch, int total_q, int total_k, int max_seqlen_q,
                           int max_seqlen_k, int H, int Hkv, int d, float scale, int causal, int deterministic,
                           void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (!cu_seqlens_q || !cu_seqlens_k) return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must not be NULL");
    return bwd_packed_impl(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, batch, total_q, max_seqlen_q, H, Hkv, d,
                           scale, causal, workspace, workspace_bytes, stream, deterministic != 0, cu_seqlens_k, total_k,
                           max_seqlen_k);
}

fa_status fa_bwd_varlen_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                      const void* dout, void* dq, void* dk, void* dv, const int* cu_seqlens,
                                      int batch, int total, int max_seqlen, int H, int Hkv, int d, float scale,
                                      int causal, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (!cu_seqlens) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must not be NULL");
    return bwd_packed_impl(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, batch, total, max_seqlen, H, Hkv, d, scale,
                           causal, workspace, workspace_bytes, stream, true);
}

fa_status fa_bwd_bnhd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int N, int H, int Hkv,
                                    int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                                    fa_stream_t stream) {
    if ((long long)B * N > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B * N exceeds the 32-bit token index");
    return bwd_packed_impl(q, k, v, o, lse, dout, dq, dk, dv, nullptr, B, B * N, N, H, Hkv, d, scale, causal,
                           workspace, workspace_bytes, stream, true);
}

fa_status fa_bwd_bnhd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                      void* dq, void* dk, void* dv, int B, int N, int H, int Hkv, int d, float scale, int causal,
                      void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    if ((long long)B * N > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B * N exceeds the 32-bit token index");
    return bwd_packed_impl(q, k, v, o, lse, dout, dq, dk, dv, nullptr, B, B * N, N, H, Hkv, d, scale, causal,
                           workspace, workspace_bytes, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    return fa_bwd_ex(FA_BF16, q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, kv_lens, workspace,
                     workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Workspace of the deterministic backward: the backward's own layout (Nq query
// rows), A - 1 more float32 dQ accumulators, the turn counters; A from the
// key blocks (Nk keys).
size_t det_workspace(int B, int H, int Hkv, int Nq, int Nk, int d) {
    const size_t base = bwd_ws_bytes(FA_BF16, B, H, Nq, d);
    if (base == 0 || Nk <= 0 || Hkv < 1 || H % Hkv != 0) return 0;
    const int nacc = det_num_acc(B, Hkv, Nk);
    return base + (size_t)(nacc - 1) * det_acc_bytes(B, H, Nq, d) + det_turn_bytes(nacc, B, H, Nq, d);
}

// Deterministic backward, square (Nk < 0), sliding window (an edge >= 0) or
// rectangular (Nk >= 0).
fa_status bwd_det_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                       void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                       int causal, int win_left, int win_right, const int* kv_lens, void* workspace,
                       size_t workspace_bytes, fa_stream_t stream, const int* row_ptr = nullptr,
                       const int* col_idx = nullptr) {
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    if (win_left < -1 || win_right < -1) return fail(FA_ERR_INVALID_ARG, "window edges must be >= -1");
    const bool rect = Nk >= 0;
    if (rect && Nk == 0) return fail(FA_ERR_INVALID_ARG, "Nk must be positive");
    const int nk = rect ? Nk : Nq;
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, Nq, d, scale, workspace, workspace_bytes, &c));
    const size_t det_need = det_workspace(B, H, Hkv, Nq, nk, d);
    const size_t need = row_ptr ? round_up(det_need, 256) + sparse_lists_bytes(Nq) : det_need;
    if (workspace_bytes < need)
        return fail(FA_ERR_INVALID_ARG, "workspace too small (%zu < %zu bytes)", workspace_bytes, need);
    const int nacc = det_num_acc(B, Hkv, nk);
    if (c.L.dqacc + det_acc_bytes(B, H, Nq, d) != c.L.total)
        return fail(FA_ERR_INVALID_ARG, "internal: the dQ accumulator is not the last workspace region");
    int* turn = reinterpret_cast<int*>(c.ws + c.L.total + (size_t)(nacc - 1) * det_acc_bytes(B, H, Nq, d));
    int *col_ptr = nullptr, *row_idx = nullptr;
    if (row_ptr) {  // block lists: transposed after the counters
        const int nb = (Nq + 127) / 128;
        col_ptr = reinterpret_cast<int*>(c.ws + round_up(det_need, 256));
        row_idx = col_ptr + nb + 1;
        cudaError_t e = fa::launch_block_lists_transpose(row_ptr, col_idx, nb, nb, col_ptr, row_idx, stream);
        if (e != cudaSuccess) return cuda_fail(e, "block list transposition launch");
    }
    FA_TRY(bwd_pre_impl(c, false, o, lse, dout, Nq, d, stream));
    FA_TRY(bwd_main_impl(c, false, q, k, v, dout, dk, dv, B, H, Nq, d, scale, causal, kv_lens, stream, Hkv, win_left,
                         win_right, col_ptr, row_idx, nullptr, 0, Nk, turn, nacc, row_ptr, col_idx));
    cudaError_t e = fa::launch_bwd_dq_det(reinterpret_cast<float*>(c.ws + c.L.dqacc), turn, dq, scale, c.BH, Nq,
                                          c.Np, d, nacc, bw_grid(c.dev), stream);
    if (e != cudaSuccess) return cuda_fail(e, "dQ conversion launch");
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_deterministic_workspace_size(int B, int H, int Hkv, int N, int d) {
    return det_workspace(B, H, Hkv, N, N, d);
}

fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                               float scale, int causal, const int* kv_lens, void* workspace, size_t workspace_bytes,
                               fa_stream_t stream) {
    return bwd_det_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, -1, d, scale, causal, -1, -1, kv_lens,
                        workspace, workspace_bytes, stream);
}

fa_status fa_bwd_window_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int N,
                                      int d, float scale, int causal, int window_left, int window_right,
                                      const int* kv_lens, void* workspace, size_t workspace_bytes,
                                      fa_stream_t stream) {
    // as fa_bwd_window: the causal mask is folded into the window's right edge
    return bwd_det_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, -1, d, scale, causal, window_left,
                        window_right, kv_lens, workspace, workspace_bytes, stream);
}

size_t fa_bwd_block_sparse_deterministic_workspace_size(int B, int H, int Hkv, int N, int d) {
    const size_t w = det_workspace(B, H, Hkv, N, N, d);
    return w ? round_up(w, 256) + sparse_lists_bytes(N) : 0;
}

fa_status fa_bwd_block_sparse_deterministic(const void* q, const void* k, const void* v, const void* o,
                                            const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                                            int H, int Hkv, int N, int d, float scale, int causal,
                                            const int* row_ptr, const int* col_idx, const int* kv_lens,
                                            void* workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (!row_ptr || !col_idx) return fail(FA_ERR_INVALID_ARG, "row_ptr and col_idx must not be NULL");
    if (N > 0 && (N + 127) / 128 > kMaxSparseBlocks)
        return fail(FA_ERR_UNSUPPORTED, "block-sparse attention takes at most %d blocks", kMaxSparseBlocks);
    return bwd_det_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, -1, d, scale, causal, -1, -1, kv_lens,
                        workspace, workspace_bytes, stream, row_ptr, col_idx);
}

size_t fa_bwd_rect_deterministic_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d) {
    return det_workspace(B, H, Hkv, Nq, Nk, d);
}

fa_status fa_bwd_rect_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq,
                                    int Nk, int d, float scale, int causal, const int* kv_lens, void* workspace,
                                    size_t workspace_bytes, fa_stream_t stream) {
    if (Nk <= 0) return fail(FA_ERR_INVALID_ARG, "Nk must be positive");
    return bwd_det_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, scale, causal, -1, -1, kv_lens,
                        workspace, workspace_bytes, stream);
}

int fa_fp8_num_blocks(int N) { return N > 0 ? (N + 63) / 64 : 0; }

fa_status fa_quantize_fp8(const void* x_bf16, void* x_e4m3, float* scales, int B, int H, int N, int d,
                          fa_stream_t stream) {
    FA_TRY(check_common(B, H, N, d, 1.0f));
    FA_CHECK_PTR(x_bf16);
    FA_CHECK_PTR(x_e4m3);
    FA_CHECK_PTR(scales);
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    fa::QuantJobs jobs;
    memset(&jobs, 0, sizeof(jobs));
    jobs.x[0] = x_bf16;
    jobs.x8[0] = x_e4m3;
    jobs.scales[0] = scales;
    jobs.heads[0] = B * H;
    cudaError_t e = fa::launch_quantize_fp8(jobs, N, d, dev->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "quantiser launch");
    return FA_OK;
}

fa_status fa_quantize_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8, float* sq,
                              float* sk, float* sv, int B, int H, int Hkv, int N, int d, fa_stream_t stream) {
    FA_TRY(check_common(B, H, N, d, 1.0f));
    if (Hkv < 1 || H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
    FA_CHECK_PTR(q);
    FA_CHECK_PTR(k);
    FA_CHECK_PTR(v);
    FA_CHECK_PTR(q8);
    FA_CHECK_PTR(k8);
    FA_CHECK_PTR(v8);
    FA_CHECK_PTR(sq);
    FA_CHECK_PTR(sk);
    FA_CHECK_PTR(sv);
    DeviceInfo* dev = nullptr;
    FA_TRY(device_info(&dev));
    const fa::QuantJobs jobs = {{q, k, v}, {q8, k8, v8}, {sq, sk, sv}, {B * H, B * Hkv, B * Hkv}};
    cudaError_t e = fa::launch_quantize_fp8(jobs, N, d, dev->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "quantiser launch");
    return FA_OK;
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk,
                     const float* sv, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
                     const int* kv_lens, fa_stream_t stream) {
    return fwd_impl(FA_BF16, 128, true, q8, k8, v8, sq, sk, sv, o, lse, B, H, N, d, scale, causal, kv_lens, nullptr, 0,
                    stream);
}

fa_status fa_fwd_fp8_gqa(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk,
                         const float* sv, void* o, float* lse, int B, int H, int Hkv, int N, int d, float scale,
                         int causal, const int* kv_lens, fa_stream_t stream) {
    return fwd_impl(FA_BF16, 128, true, q8, k8, v8, sq, sk, sv, o, lse, B, H, N, d, scale, causal, kv_lens, nullptr, 0,
                    stream, 1, nullptr, 0, Hkv);
}

fa_status fa_fwd_fp8_split(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk,
                           const float* sv, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
                           const int* kv_lens, int num_splits, void* workspace, size_t workspace_bytes,
                           fa_stream_t stream) {
    return fwd_impl(FA_BF16, 128, true, q8, k8, v8, sq, sk, sv, o, lse, B, H, N, d, scale, causal, kv_lens, nullptr, 0,
                    stream, num_splits, workspace, workspace_bytes);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// FP8 backward (chapter 18 §18.6.2: FP8 tensor-core products, dS in E5M2,
// float32 gradients).  Workspace: the bf16 backward's layout (statistics,
// float32 dQ accumulator), then dO's E4M3 codes and block scales, then K8
// transposed ([B*H][128][Np] codes) for the dQ product's K-major operand.
// ---------------------------------------------------------------------------
namespace {

struct Fp8BwdLayout {
    size_t base, do8, sdo, kt, total;
};
Fp8BwdLayout fp8_bwd_layout(int B, int H, int N) {
    const size_t BH = (size_t)B * H, Np = round_up((size_t)N, 128), nblk = (N + 63) / 64;
    Fp8BwdLayout L;
    L.base = 0;
    size_t off = round_up(bwd_ws_bytes(FA_BF16, B, H, N, 128), 256);
    L.do8 = off; off = round_up(off + BH * N * 128, 256);
    L.sdo = off; off = round_up(off + BH * nblk * 4, 256);
    L.kt = off; off = round_up(off + BH * 128 * Np, 256);
    L.total = off;
    return L;
}

fa_status bwd_fp8_impl(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk,
                       const float* sv, const void* o, const float* lse, const void* dout, float* dq, float* dk,
                       float* dv, int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    FA_CHECK_PTR(q8);
    FA_CHECK_PTR(k8);
    FA_CHECK_PTR(v8);
    FA_CHECK_PTR(sq);
    FA_CHECK_PTR(sk);
    FA_CHECK_PTR(sv);
    FA_CHECK_PTR(o);
    FA_CHECK_PTR(lse);
    FA_CHECK_PTR(dout);
    FA_CHECK_PTR(dq);
    FA_CHECK_PTR(dk);
    FA_CHECK_PTR(dv);
    if (d != 128) return fail(FA_ERR_UNSUPPORTED, "the FP8 backward needs d = 128");
    BwdCtx c{};
    FA_TRY(bwd_setup(FA_BF16, B, H, N, d, scale, workspace, workspace_bytes, &c));
    const Fp8BwdLayout L = fp8_bwd_layout(B, H, N);
    if (workspace_bytes < L.total)
        return fail(FA_ERR_INVALID_ARG, "workspace too small (%zu < %zu bytes)", workspace_bytes, L.total);
    const int nblk = (N + 63) / 64, BH = c.BH, Np = c.Np;
    uint8_t* do8 = reinterpret_cast<uint8_t*>(c.ws + L.do8);
    float* sdo = reinterpret_cast<float*>(c.ws + L.sdo);
    uint8_t* kt = reinterpret_cast<uint8_t*>(c.ws + L.kt);
    // dO8; D = rowsum(dO^ * O) from the dequantised dO8, LSE * log2(e), zeroed
    // accumulator; K8 transposed
    fa::QuantJobs jobs;
    memset(&jobs, 0, sizeof(jobs));
    jobs.x[0] = dout;
    jobs.x8[0] = do8;
    jobs.scales[0] = sdo;
    jobs.heads[0] = BH;
    cudaError_t e = fa::launch_quantize_fp8(jobs, N, d, c.dev->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "dO quantiser launch");
    e = fa::launch_bwd_pre_fp8(o, do8, sdo, lse, reinterpret_cast<float*>(c.ws + c.L.lse2),
                               reinterpret_cast<float*>(c.ws + c.L.dvec), reinterpret_cast<float*>(c.ws + c.L.dqacc),
                               BH, N, Np, bw_grid(c.dev), stream);
    if (e != cudaSuccess) return cuda_fail(e, "FP8 backward preprocess launch");
    e = fa::launch_transpose_k8(k8, kt, BH, N, Np, c.dev->sms * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "K transpose launch");
    CUtensorMap tq, tk, tv, tdo, tkt, tdq;
    const auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    FA_TRY(make_map_3d(&tq, U8, 1, q8, 128, N, BH, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tk, U8, 1, k8, 128, N, BH, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tv, U8, 1, v8, 128, N, BH, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tdo, U8, 1, do8, 128, N, BH, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    FA_TRY(make_map_3d(&tkt, U8, 1, kt, Np, 128, BH, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B));
    float* dqacc = reinterpret_cast<float*>(c.ws + c.L.dqacc);
    if ((long long)BH * Np >= (1LL << 31))
        return fail(FA_ERR_UNSUPPORTED, "dQ accumulator rows exceed the 32-bit tensor coordinate range");
    FA_TRY(make_map_dqacc(&tdq, dqacc, d, (long long)BH * Np, 128));
    fa::BwdFp8Params p;
    memset(&p, 0, sizeof(p));
    p.B = B; p.H = H; p.N = N; p.Np = Np; p.nblk = nblk;
    p.num_kt = (N + 127) / 128;
    p.num_items = BH * p.num_kt;
    p.causal = causal != 0;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kv_lens = kv_lens;
    p.sq = sq; p.sk = sk; p.sv = sv; p.sdo = sdo;
    p.lse2 = reinterpret_cast<float*>(c.ws + c.L.lse2);
    p.dvec = reinterpret_cast<float*>(c.ws + c.L.dvec);
    p.dk = dk;
    p.dv = dv;
    p.err = c.dev->err_word;
    e = fa::launch_bwd_fp8(tq, tk, tv, tdo, tkt, tdq, p, grid_for_items(p.num_items, c.dev->sms), stream);
    if (e != cudaSuccess) return cuda_fail(e, "FP8 backward launch");
    return bwd_dq_impl(c, true, dq, N, d, scale, stream);
}

}  // namespace

// ---------------------------------------------------------------------------
// One call per pass: the parameter block of include/fa.h.  attn_plan is the one
// validation routine of both passes: it names the kernel family a parameter
// block selects, or refuses the combination (before any launch) with the
// reason; the entry points then call that family's implementation above.
// ---------------------------------------------------------------------------
namespace {

enum class Family {
    Plain,        // [B,H,N,d] bf16, N_q = N_k, H = Hkv, no window / lists
    F32,          // float32 tensors
    Gqa,          // shared key/value heads
    Window,       // sliding window
    Sparse,       // block lists
    Rect,         // N_q != N_k
    Packed,       // packed sequences (optionally windowed)
    PackedKv,     // packed sequences with their own key ranges
    Bnhd,         // flash_attn_func's [B, N, H, d]
    Fp8,          // E4M3 inputs
};

struct AttnPlan {
    Family fam;
    int Hkv, Nk, total_k;
    bool window, det;
};

fa_status attn_plan(const fa_attn_params* a, bool bwd, AttnPlan* pl) {
    if (!a) return fail(FA_ERR_INVALID_ARG, "params must not be NULL");
    if (a->struct_size != sizeof(fa_attn_params))
        return fail(FA_ERR_INVALID_ARG,
                    "params->struct_size is %zu, this library's fa_attn_params has %zu bytes (initialise it with "
                    "fa_attn_params_init from the same header version)",
                    a->struct_size, sizeof(fa_attn_params));
    if (a->heads <= 0 || a->batch <= 0 || a->seqlen_q <= 0)
        return fail(FA_ERR_INVALID_ARG, "batch, heads and seqlen_q must be positive");
    const int Hkv = a->kv_heads ? a->kv_heads : a->heads;
    if (Hkv < 1 || a->heads % Hkv != 0)
        return fail(FA_ERR_INVALID_ARG, "heads (%d) must be a multiple of kv_heads (%d)", a->heads, Hkv);
    if (a->window_left < -1 || a->window_right < -1)
        return fail(FA_ERR_INVALID_ARG, "window edges must be >= -1 (-1 = unbounded)");
    if (a->seqlen_k < 0 || a->num_splits < 0 || a->block_c < 0)
        return fail(FA_ERR_INVALID_ARG, "seqlen_k, num_splits and block_c must be >= 0");
    if ((a->block_row_ptr == nullptr) != (a->block_col_idx == nullptr))
        return fail(FA_ERR_INVALID_ARG, "block lists need both block_row_ptr and block_col_idx");
    pl->Hkv = Hkv;
    pl->Nk = a->seqlen_k ? a->seqlen_k : a->seqlen_q;
    pl->total_k = a->total_k ? a->total_k : a->total_q;
    pl->window = a->window_left >= 0 || a->window_right >= 0;
    pl->det = a->deterministic != 0;
    // a nonzero seqlen_k selects the rectangular kernels (also when it equals seqlen_q)
    const bool sparse = a->block_row_ptr != nullptr, rect = a->seqlen_k != 0;
    const bool split = a->num_splits != 1;
    auto refuse = [](const char* what) { return fail(FA_ERR_UNSUPPORTED, "not built: %s", what); };
    if (bwd && (a->num_splits > 1 || a->block_c)) return refuse("num_splits / block_c in a backward call");
    if (!bwd && pl->det) return refuse("deterministic in a forward call");
    switch (a->dtype) {
    case FA_E4M3:
        if (a->layout != FA_LAYOUT_BHND || pl->window || sparse || rect)
            return refuse("FP8 with the packed or [B,N,H,d] layouts, a window, block lists or N_q != N_k");
        if (bwd && (Hkv != a->heads || pl->det)) return refuse("the FP8 backward with shared key/value heads or "
                                                               "deterministic");
        if (Hkv != a->heads && split) return refuse("a split FP8 forward with shared key/value heads");
        if (a->block_c) return refuse("block_c with FP8");
        pl->fam = Family::Fp8;
        return FA_OK;
    case FA_F32:
        if (a->layout != FA_LAYOUT_BHND || pl->window || sparse || rect || Hkv != a->heads || split || pl->det)
            return refuse("float32 tensors with options beyond causal, kv_lens and block_c");
        pl->fam = Family::F32;
        return FA_OK;
    case FA_BF16:
        break;
    default:
        return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)a->dtype);
    }
    if (a->layout == FA_LAYOUT_PACKED) {
        if (!a->cu_seqlens_q) return fail(FA_ERR_INVALID_ARG, "the packed layout needs cu_seqlens_q");
        if (a->kv_lens || sparse || split || a->block_c)
            return refuse("kv_lens, block lists, num_splits or block_c with the packed layout");
        if (a->total_q <= 0) return fail(FA_ERR_INVALID_ARG, "the packed layout needs total_q > 0");
        if (a->cu_seqlens_k) {
            if (pl->window) return refuse("a window with separate packed key ranges");
            pl->fam = Family::PackedKv;
        } else {
            pl->fam = Family::Packed;
        }
        return FA_OK;
    }
    if (a->layout == FA_LAYOUT_BNHD) {
        if (a->kv_lens || sparse || pl->window || rect || split || a->block_c)
            return refuse("kv_lens, block lists, a window, N_q != N_k, num_splits or block_c with the [B,N,H,d] "
                          "layout (packed sequences cover different lengths)");
        pl->fam = Family::Bnhd;
        return FA_OK;
    }
    if (a->layout != FA_LAYOUT_BHND) return fail(FA_ERR_INVALID_ARG, "unknown layout %d", (int)a->layout);
    if (rect) {
        if (pl->window || sparse || a->block_c) return refuse("a window, block lists or block_c with N_q != N_k");
        pl->fam = Family::Rect;
        return FA_OK;
    }
    if (sparse) {
        if (pl->window || split || a->block_c) return refuse("block lists with a window, num_splits or block_c");
        pl->fam = Family::Sparse;
        return FA_OK;
    }
    if (pl->window) {
        if (split || a->block_c) return refuse("a window with num_splits or block_c");
        pl->fam = Family::Window;
        return FA_OK;
    }
    if (Hkv != a->heads) {
        if (split || a->block_c) return refuse("shared key/value heads with num_splits or block_c");
        pl->fam = Family::Gqa;
        return FA_OK;
    }
    if (split && a->block_c) return refuse("num_splits with block_c");
    pl->fam = Family::Plain;
    return FA_OK;
}

}  // namespace

extern "C" {

void fa_attn_params_init(fa_attn_params* p) {
    if (!p) return;
    memset(p, 0, sizeof(*p));
    p->struct_size = sizeof(fa_attn_params);
    p->dtype = FA_BF16;
    p->layout = FA_LAYOUT_BHND;
    p->window_left = p->window_right = -1;
    p->num_splits = 1;
}

size_t fa_attn_fwd_workspace_size(const fa_attn_params* a) {
    AttnPlan pl;
    if (attn_plan(a, false, &pl) != FA_OK) return 0;
    const int B = a->batch, H = a->heads, N = a->seqlen_q, d = a->head_dim;
    switch (pl.fam) {
    case Family::Plain:
    case Family::Fp8:
        return fa_fwd_split_workspace_size(B, H, N, d, a->causal, a->kv_lens != nullptr, a->num_splits);
    case Family::Rect:
        return fa_fwd_rect_workspace_size(B, H, pl.Hkv, N, pl.Nk, d, a->num_splits);
    case Family::F32:
        return fa_fwd_workspace_size(FA_F32, B, H, N, d);
    default:
        return 0;
    }
}

int fa_attn_fwd_splits(const fa_attn_params* a) {
    AttnPlan pl;
    if (attn_plan(a, false, &pl) != FA_OK) return 1;
    const int B = a->batch, H = a->heads, N = a->seqlen_q, d = a->head_dim;
    if (pl.fam == Family::Plain || pl.fam == Family::Fp8)
        return fa_fwd_split_count(B, H, N, d, a->causal, a->kv_lens != nullptr, a->num_splits);
    if (pl.fam == Family::Rect) return fa_fwd_rect_split_count(B, H, pl.Hkv, N, pl.Nk, d, a->num_splits);
    return 1;
}

size_t fa_attn_bwd_workspace_size(const fa_attn_params* a) {
    AttnPlan pl;
    if (attn_plan(a, true, &pl) != FA_OK) return 0;
    const int B = a->batch, H = a->heads, N = a->seqlen_q, d = a->head_dim, Hkv = pl.Hkv;
    switch (pl.fam) {
    case Family::Plain:
        return pl.det ? fa_bwd_deterministic_workspace_size(B, H, Hkv, N, d) : bwd_ws_bytes(FA_BF16, B, H, N, d);
    case Family::F32:
        return bwd_ws_bytes(FA_F32, B, H, N, d);
    case Family::Gqa:
        return pl.det ? fa_bwd_deterministic_workspace_size(B, H, Hkv, N, d) : fa_bwd_gqa_workspace_size(B, H, Hkv, N, d);
    case Family::Window:
        return pl.det ? fa_bwd_deterministic_workspace_size(B, H, Hkv, N, d) : fa_bwd_gqa_workspace_size(B, H, Hkv, N, d);
    case Family::Sparse:
        return pl.det ? fa_bwd_block_sparse_deterministic_workspace_size(B, H, Hkv, N, d)
                      : fa_bwd_block_sparse_workspace_size(B, H, N, d);
    case Family::Rect:
        return pl.det ? fa_bwd_rect_deterministic_workspace_size(B, H, Hkv, N, pl.Nk, d)
                      : fa_bwd_rect_workspace_size(B, H, Hkv, N, pl.Nk, d);
    case Family::Packed:
        return pl.det ? fa_bwd_varlen_deterministic_workspace_size(B, N, H, Hkv, d) : fa_bwd_varlen_workspace_size(B, N, H, d);
    case Family::PackedKv:
        return fa_bwd_varlen_kv_workspace_size(B, N, a->seqlen_k ? a->seqlen_k : N, H, Hkv, d, a->deterministic);
    case Family::Bnhd:
        return pl.det ? fa_bwd_bnhd_deterministic_workspace_size(B, N, H, Hkv, d) : fa_bwd_bnhd_workspace_size(B, N, H, d);
    case Family::Fp8:
        return d == 128 ? fp8_bwd_layout(B, H, N).total : 0;
    default:
        return 0;
    }
}

fa_status fa_attn_fwd(const fa_attn_params* a, fa_stream_t stream) {
    AttnPlan pl;
    FA_TRY(attn_plan(a, false, &pl));
    const int B = a->batch, H = a->heads, N = a->seqlen_q, d = a->head_dim, Hkv = pl.Hkv;
    switch (pl.fam) {
    case Family::Plain:
        if (a->block_c)
            return fa_fwd_ex(FA_BF16, a->block_c, a->q, a->k, a->v, a->o, a->lse, B, H, N, d, a->scale, a->causal,
                             a->kv_lens, nullptr, 0, stream);
        return fa_fwd_split(a->q, a->k, a->v, a->o, a->lse, B, H, N, d, a->scale, a->causal, a->kv_lens, a->num_splits,
                            a->workspace, a->workspace_bytes, stream);
    case Family::F32:
        return fa_fwd_ex(FA_F32, a->block_c, a->q, a->k, a->v, a->o, a->lse, B, H, N, d, a->scale, a->causal,
                         a->kv_lens, a->workspace, a->workspace_bytes, stream);
    case Family::Gqa:
        return fa_fwd_gqa(a->q, a->k, a->v, a->o, a->lse, B, H, Hkv, N, d, a->scale, a->causal, a->kv_lens, stream);
    case Family::Window:
        return fa_fwd_window(a->q, a->k, a->v, a->o, a->lse, B, H, Hkv, N, d, a->scale, a->causal, a->window_left,
                             a->window_right, a->kv_lens, stream);
    case Family::Sparse:
        return fa_fwd_block_sparse(a->q, a->k, a->v, a->o, a->lse, B, H, Hkv, N, d, a->scale, a->causal,
                                   a->block_row_ptr, a->block_col_idx, a->kv_lens, stream);
    case Family::Rect:
        return fa_fwd_rect(a->q, a->k, a->v, a->o, a->lse, B, H, Hkv, N, pl.Nk, d, a->scale, a->causal, a->kv_lens,
                           a->num_splits, a->workspace, a->workspace_bytes, stream);
    case Family::Packed:
        if (pl.window)
            return fa_fwd_varlen_window(a->q, a->k, a->v, a->o, a->lse, a->cu_seqlens_q, B, a->total_q, N, H, Hkv, d,
                                        a->scale, a->causal, a->window_left, a->window_right, stream);
        return fa_fwd_varlen(a->q, a->k, a->v, a->o, a->lse, a->cu_seqlens_q, B, a->total_q, N, H, Hkv, d, a->scale,
                             a->causal, stream);
    case Family::PackedKv:
        return fa_fwd_varlen_kv(a->q, a->k, a->v, a->o, a->lse, a->cu_seqlens_q, a->cu_seqlens_k, B, a->total_q,
                                pl.total_k, N, H, Hkv, d, a->scale, a->causal, stream);
    case Family::Bnhd:
        return fa_fwd_bnhd(a->q, a->k, a->v, a->o, a->lse, B, N, H, Hkv, d, a->scale, a->causal, stream);
    case Family::Fp8:
        if (Hkv != H)
            return fa_fwd_fp8_gqa(a->q, a->k, a->v, a->q_scale, a->k_scale, a->v_scale, a->o, a->lse, B, H, Hkv, N, d,
                                  a->scale, a->causal, a->kv_lens, stream);
        return fa_fwd_fp8_split(a->q, a->k, a->v, a->q_scale, a->k_scale, a->v_scale, a->o, a->lse, B, H, N, d,
                                a->scale, a->causal, a->kv_lens, a->num_splits, a->workspace, a->workspace_bytes,
                                stream);
    }
    return fail(FA_ERR_INVALID_ARG, "internal: unknown kernel family");
}

fa_status fa_attn_bwd(const fa_attn_params* a, fa_stream_t stream) {
    AttnPlan pl;
    FA_TRY(attn_plan(a, true, &pl));
    const int B = a->batch, H = a->heads, N = a->seqlen_q, d = a->head_dim, Hkv = pl.Hkv;
    const bool det = pl.det;
    void* ws = a->workspace;
    const size_t wsb = a->workspace_bytes;
    switch (pl.fam) {
    case Family::Plain:
        if (det)
            return fa_bwd_deterministic(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, B, H, H, N, d,
                                        a->scale, a->causal, a->kv_lens, ws, wsb, stream);
        return fa_bwd(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, B, H, N, d, a->scale, a->causal,
                      a->kv_lens, ws, wsb, stream);
    case Family::F32:
        return fa_bwd_ex(FA_F32, a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, B, H, N, d, a->scale,
                         a->causal, a->kv_lens, ws, wsb, stream);
    case Family::Gqa:
        if (det)
            return fa_bwd_deterministic(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, B, H, Hkv, N, d,
                                        a->scale, a->causal, a->kv_lens, ws, wsb, stream);
        return fa_bwd_gqa(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, B, H, Hkv, N, d, a->scale,
                          a->causal, a->kv_lens, ws, wsb, stream);
    case Family::Window:
        return (det ? fa_bwd_window_deterministic : fa_bwd_window)(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq,
                                                                   a->dk, a->dv, B, H, Hkv, N, d, a->scale, a->causal,
                                                                   a->window_left, a->window_right, a->kv_lens, ws,
                                                                   wsb, stream);
    case Family::Sparse:
        return (det ? fa_bwd_block_sparse_deterministic : fa_bwd_block_sparse)(
            a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, B, H, Hkv, N, d, a->scale, a->causal,
            a->block_row_ptr, a->block_col_idx, a->kv_lens, ws, wsb, stream);
    case Family::Rect:
        return (det ? fa_bwd_rect_deterministic : fa_bwd_rect)(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk,
                                                               a->dv, B, H, Hkv, N, pl.Nk, d, a->scale, a->causal,
                                                               a->kv_lens, ws, wsb, stream);
    case Family::Packed:
        if (pl.window)
            return fa_bwd_varlen_window(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, a->cu_seqlens_q,
                                        B, a->total_q, N, H, Hkv, d, a->scale, a->causal, a->window_left,
                                        a->window_right, a->deterministic, ws, wsb, stream);
        return (det ? fa_bwd_varlen_deterministic : fa_bwd_varlen)(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq,
                                                                   a->dk, a->dv, a->cu_seqlens_q, B, a->total_q, N, H,
                                                                   Hkv, d, a->scale, a->causal, ws, wsb, stream);
    case Family::PackedKv:
        return fa_bwd_varlen_kv(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk, a->dv, a->cu_seqlens_q,
                                a->cu_seqlens_k, B, a->total_q, pl.total_k, N, a->seqlen_k ? a->seqlen_k : N, H, Hkv,
                                d, a->scale, a->causal, a->deterministic, ws, wsb, stream);
    case Family::Bnhd:
        return (det ? fa_bwd_bnhd_deterministic : fa_bwd_bnhd)(a->q, a->k, a->v, a->o, a->lse, a->dout, a->dq, a->dk,
                                                               a->dv, B, N, H, Hkv, d, a->scale, a->causal, ws, wsb,
                                                               stream);
    case Family::Fp8:
        return bwd_fp8_impl(a->q, a->k, a->v, a->q_scale, a->k_scale, a->v_scale, a->o, a->lse, a->dout,
                            reinterpret_cast<float*>(a->dq), reinterpret_cast<float*>(a->dk),
                            reinterpret_cast<float*>(a->dv), B, H, N, d, a->scale, a->causal, a->kv_lens, ws, wsb,
                            stream);
    }
    return fail(FA_ERR_INVALID_ARG, "internal: unknown kernel family");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free backward.
//
// Some callers of this library cannot allocate device memory at all: for
// example a plugin hosted inside a framework that owns the whole device-memory
// pool and offers it no allocation hook, or a runtime that forbids allocation
// once it has started so that its latency stays predictable.  For them the
// backward's scratch (the row statistics and the float32 dQ accumulator) lives
// in a fixed array of device memory that this library defines below; every GPU
// that loads the library keeps it until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 128ull << 20;  // 128 MiB

static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, looked up once per device (with that
// device current).  In host code the array's name is only a stand-in symbol,
// never a device address, so it is never passed to a kernel directly.
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

fa_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fa_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const int* kv_lens, fa_stream_t stream) {
    FA_TRY(check_common(B, H, N, d, scale));
    const size_t need = bwd_ws_bytes(FA_BF16, B, H, N, d);
    if (need > kNoAllocScratchBytes)
        return fail(FA_ERR_INVALID_ARG,
                    "fa_bwd_noalloc: this problem needs %zu bytes of scratch, more than the %zu-byte static array; "
                    "use fa_bwd with a caller-provided workspace",
                    need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    FA_TRY(noalloc_scratch(&scratch));
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, kv_lens, scratch,
                  kNoAllocScratchBytes, stream);
}

}  // extern "C"

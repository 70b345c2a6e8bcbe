// Bandwidth-bound kernels around the two tensor-core kernels:
//   * backward preprocess: D_i = rowsum(dO_i * O_i) (FA-v2 analysis page §5.2,
//     attention-kernels wiki §04 "D_i = G_i . O_i"), the saved LSE moved to the
//     log2 domain (+inf on rows with no visible key and on padding rows, so
//     the backward's P is exactly 0 there), and the zeroed float32 dQ
//     accumulator;
//   * dQ conversion: dQ = scale * dQ_acc (the 1/sqrt(d) of wiki §04);
//   * FP8 E4M3 per-block quantiser (chapter 18 §18.6.2: s = max|X| / 448);
//   * float32 -> bf16 rounding of inputs for the float32 entry points;
//   * the merge of the split-key forward's partial results (chapter 18
//     §18.8.2, FlashDecoding: the reduction that combines the per-range
//     statistics and outputs with the online-softmax weights).
// All use 16-byte vector accesses and grid-stride loops over a grid sized in
// multiples of the SM count.
#include <cuda_bf16.h>
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// L2 eviction priorities for the backward's streaming kernels.  The
// preprocess reads O and dO once (evict first) and zeroes the float32 dQ
// accumulator with evict-last stores, so that the zeroed lines are still in
// L2 when the main kernel's bulk additions reach them; the dQ conversion reads
// the accumulator for the last time (evict first).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// 16-byte read-only load that skips L1, with an L2 eviction policy
__device__ __forceinline__ uint4 ld_stream(const void* ptr, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr), "l"(pol));
    return v;
}
// 16 zero bytes, with an L2 eviction policy
__device__ __forceinline__ void st_keep_zero(void* ptr, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %1, %1, %1}, %2;" :: "l"(ptr), "r"(0u), "l"(pol) : "memory");
}

// One group of LPR lanes per row; each lane covers 8 consecutive elements.
template <int D, bool IN_F32>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const void* __restrict__ o, const void* __restrict__ dout,
                                                      const float* __restrict__ lse, float* __restrict__ lse2,
                                                      float* __restrict__ dvec, float* __restrict__ dq_acc, int BH,
                                                      int N, int Np) {
    constexpr int LPR = D / 8;                 // lanes per row
    constexpr int RPW = 32 / LPR;              // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, sl = lane % LPR;
    const long total_rows = (long)BH * Np;
    const long warps = (long)gridDim.x * (blockDim.x / 32);
    const long gw = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    for (long r0 = gw * RPW; r0 < total_rows; r0 += warps * RPW) {
        const long r = r0 + sub;
        const bool valid_row = r < total_rows;
        const long bh = valid_row ? r / Np : 0;
        const int i = valid_row ? (int)(r - bh * Np) : 0;
        float acc = 0.f;
        if (valid_row && i < N) {
            const size_t e = ((size_t)bh * N + i) * D + sl * 8;
            float a[8], b[8];
            if constexpr (IN_F32) {
                const float4* po = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(o) + e);
                const float4* pg = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(dout) + e);
                const float4 o0 = __ldg(po), o1 = __ldg(po + 1), g0 = __ldg(pg), g1 = __ldg(pg + 1);
                a[0] = o0.x; a[1] = o0.y; a[2] = o0.z; a[3] = o0.w; a[4] = o1.x; a[5] = o1.y; a[6] = o1.z; a[7] = o1.w;
                b[0] = g0.x; b[1] = g0.y; b[2] = g0.z; b[3] = g0.w; b[4] = g1.x; b[5] = g1.y; b[6] = g1.z; b[7] = g1.w;
            } else {
                unpack8(ld_stream(reinterpret_cast<const __nv_bfloat16*>(o) + e, pol_first), a);
                unpack8(ld_stream(reinterpret_cast<const __nv_bfloat16*>(dout) + e, pol_first), b);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) acc = fmaf(a[k], b[k], acc);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid_row) {
            float* qa = dq_acc + (size_t)r * D + sl * 8;
            st_keep_zero(qa, pol_last);
            st_keep_zero(qa + 4, pol_last);
            if (sl == 0) {
                float l2 = INFINITY;
                if (i < N) {
                    const float L = lse[(size_t)bh * N + i];
                    l2 = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
                }
                lse2[r] = l2;
                dvec[r] = (i < N) ? acc : 0.f;
            }
        }
    }
}

// The FP8 backward's preprocess (d = 128): D = rowsum(dO^ * O) with dO^ the
// dequantised E4M3 upstream gradient s_do * dO8 the backward's products use
// (so that D matches their dP = dO^ V^T), LSE * log2(e), and the zeroed dQ
// accumulator.  One group of 16 lanes per row; 8 elements per lane.
__global__ void __launch_bounds__(256) bwd_pre_fp8_kernel(const __nv_bfloat16* __restrict__ o,
                                                          const uint8_t* __restrict__ do8,
                                                          const float* __restrict__ sdo, const float* __restrict__ lse,
                                                          float* __restrict__ lse2, float* __restrict__ dvec,
                                                          float* __restrict__ dq_acc, int BH, int N, int Np, int nblk) {
    constexpr int D = 128, LPR = 16, RPW = 2;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, sl = lane % LPR;
    const long total_rows = (long)BH * Np;
    const long warps = (long)gridDim.x * (blockDim.x / 32);
    const long gw = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
    const uint64_t pol_first = policy_evict_first(), pol_last = policy_evict_last();
    for (long r0 = gw * RPW; r0 < total_rows; r0 += warps * RPW) {
        const long r = r0 + sub;
        const bool valid_row = r < total_rows;
        const long bh = valid_row ? r / Np : 0;
        const int i = valid_row ? (int)(r - bh * Np) : 0;
        float acc = 0.f;
        if (valid_row && i < N) {
            const size_t e = ((size_t)bh * N + i) * D + sl * 8;
            float a[8];
            unpack8(ld_stream(o + e, pol_first), a);
            const uint2 c = *reinterpret_cast<const uint2*>(do8 + e);
            const float s = __ldg(sdo + bh * nblk + i / 64);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float2 g = __half22float2(e4m3x2_to_half2(((h < 2 ? c.x : c.y) >> (16 * (h & 1))) & 0xFFFFu));
                acc = fmaf(a[2 * h], g.x * s, acc);
                acc = fmaf(a[2 * h + 1], g.y * s, acc);
            }
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid_row) {
            float* qa = dq_acc + (size_t)r * D + sl * 8;
            st_keep_zero(qa, pol_last);
            st_keep_zero(qa + 4, pol_last);
            if (sl == 0) {
                float l2 = INFINITY;
                if (i < N) {
                    const float L = lse[(size_t)bh * N + i];
                    l2 = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
                }
                lse2[r] = l2;
                dvec[r] = (i < N) ? acc : 0.f;
            }
        }
    }
}

// dQ[r, :] = scale * dQ_acc[r, :] for the N real rows of every head.  Each
// thread converts U 8-element groups per pass, all loads issued before the
// stores, so that enough reads stay in flight to keep HBM busy.
template <bool OUT_F32>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc, void* __restrict__ dq, float scale,
                                                     int BH, int N, int Np, int D) {
    constexpr int U = 4;
    const long groups_per_row = D / 8;
    const long total = (long)BH * N * groups_per_row;
    const long stride = (long)gridDim.x * blockDim.x;
    const uint64_t pol_first = policy_evict_first();
    for (long g0 = (long)blockIdx.x * blockDim.x + threadIdx.x; g0 < total; g0 += U * stride) {
        float4 a[U], b[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long g = g0 + u * stride;
            if (g >= total) continue;
            const long row = g / groups_per_row;
            const int c = (int)(g - row * groups_per_row) * 8;
            const long bh = row / N;
            const long i = row - bh * N;
            const float4* src = reinterpret_cast<const float4*>(acc + ((size_t)bh * Np + i) * D + c);
            const uint4 ua = ld_stream(src, pol_first), ub = ld_stream(src + 1, pol_first);
            a[u] = make_float4(__uint_as_float(ua.x), __uint_as_float(ua.y), __uint_as_float(ua.z), __uint_as_float(ua.w));
            b[u] = make_float4(__uint_as_float(ub.x), __uint_as_float(ub.y), __uint_as_float(ub.z), __uint_as_float(ub.w));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long g = g0 + u * stride;
            if (g >= total) continue;
            const size_t e = (size_t)g * 8;  // row * D + c
            if constexpr (OUT_F32) {
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(dq) + e);
                dst[0] = make_float4(a[u].x * scale, a[u].y * scale, a[u].z * scale, a[u].w * scale);
                dst[1] = make_float4(b[u].x * scale, b[u].y * scale, b[u].z * scale, b[u].w * scale);
            } else {
                *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dq) + e) = make_uint4(
                    pack_bf16x2(a[u].x * scale, a[u].y * scale), pack_bf16x2(a[u].z * scale, a[u].w * scale),
                    pack_bf16x2(b[u].x * scale, b[u].y * scale), pack_bf16x2(b[u].z * scale, b[u].w * scale));
            }
        }
    }
}

// Deterministic backward's conversion: dQ[r, :] = scale * the sum, in order
// a = 0, 1, ..., of the accumulators a that received a write for row r's
// quarter of its tile (turn count > 0; the others were never written).  Tiles
// are BR = 64 rows with quarters of 32 columns (d = 128), or BR = 128 rows with
// quarters of 32 rows (d = 64).
__global__ void __launch_bounds__(256) bwd_dq_det_kernel(const float* __restrict__ acc, const int* __restrict__ turn,
                                                         __nv_bfloat16* __restrict__ dq, float scale, int BH, int N,
                                                         int Np, int D, int nacc) {
    constexpr int kMaxAcc = 8;
    const int BR = (D == 128) ? 64 : 128, nqb = Np / BR;
    const long groups_per_row = D / 8;
    const long total = (long)BH * N * groups_per_row;
    const size_t acc_elems = (size_t)BH * Np * D, turn_stride = (size_t)BH * nqb * 4;
    for (long g = (long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (long)gridDim.x * blockDim.x) {
        const long row = g / groups_per_row;
        const int c = (int)(g - row * groups_per_row) * 8;
        const long bh = row / N;
        const int i = (int)(row - bh * N);
        const int quarter = (D == 128) ? c / 32 : (i % 128) / 32;
        const size_t tix = ((size_t)bh * nqb + i / BR) * 4 + quarter;
        const size_t off = ((size_t)bh * Np + i) * D + c;
        // all counts, then all written accumulators, as independent loads
        bool has[kMaxAcc];
#pragma unroll
        for (int a = 0; a < kMaxAcc; ++a) has[a] = a < nacc && __ldg(turn + a * turn_stride + tix) != 0;
        float4 x[kMaxAcc], y[kMaxAcc];
#pragma unroll
        for (int a = 0; a < kMaxAcc; ++a) {
            if (has[a]) {
                const float4* src = reinterpret_cast<const float4*>(acc + a * acc_elems + off);
                x[a] = __ldg(src);
                y[a] = __ldg(src + 1);
            }
        }
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < kMaxAcc; ++a) {
            if (has[a]) {
                s[0] += x[a].x; s[1] += x[a].y; s[2] += x[a].z; s[3] += x[a].w;
                s[4] += y[a].x; s[5] += y[a].y; s[6] += y[a].z; s[7] += y[a].w;
            }
        }
        *reinterpret_cast<uint4*>(dq + (size_t)row * D + c) =
            make_uint4(pack_bf16x2(s[0] * scale, s[1] * scale), pack_bf16x2(s[2] * scale, s[3] * scale),
                       pack_bf16x2(s[4] * scale, s[5] * scale), pack_bf16x2(s[6] * scale, s[7] * scale));
    }
}

// Packed variable-length sequences: the statistics and the dQ accumulator are
// laid out per (head, sequence) as [H][batch][MSp] rows (MSp = max_seqlen
// rounded up to 128), so that every query block of every sequence starts on
// an aligned row and padding rows (position >= the sequence's length) carry
// LSE*log2(e) = +inf, D = 0 (their P is 0 in the backward).  Row r = (h *
// batch + b) * MSp + pos reads token cu_seqlens[b] + pos of O, dO [total, H, d].
// Without cu_seqlens every sequence has max_seqlen tokens (token b *
// max_seqlen + pos: [B, N, H, d] tensors) and the LSE is [B, H, N].
__device__ __forceinline__ int varlen_len(const int* cu, int b, int max_seqlen) {
    return cu ? max(0, min(__ldg(cu + b + 1) - __ldg(cu + b), max_seqlen)) : max_seqlen;
}
__device__ __forceinline__ long varlen_token(const int* cu, int b, int max_seqlen, int pos) {
    return (cu ? (long)__ldg(cu + b) : (long)b * max_seqlen) + pos;
}

template <int D>
__global__ void __launch_bounds__(256) bwd_pre_varlen_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse, const int* __restrict__ cu,
                                                             float* __restrict__ lse2, float* __restrict__ dvec,
                                                             float* __restrict__ dq_acc, int H, int batch, int total,
                                                             int max_seqlen, int MSp) {
    constexpr int LPR = D / 8;     // lanes per row
    constexpr int RPW = 32 / LPR;  // rows per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, sl = lane % LPR;
    const long total_rows = (long)H * batch * MSp;
    const long warps = (long)gridDim.x * (blockDim.x / 32);
    const long gw = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
    for (long r0 = gw * RPW; r0 < total_rows; r0 += warps * RPW) {
        const long r = r0 + sub;
        const bool valid_row = r < total_rows;
        const long hb = valid_row ? r / MSp : 0;
        const int pos = valid_row ? (int)(r - hb * MSp) : 0;
        const int h = (int)(hb / batch), b = (int)(hb - (long)h * batch);
        const bool real = valid_row && pos < varlen_len(cu, b, max_seqlen);
        const long token = real ? varlen_token(cu, b, max_seqlen, pos) : 0;
        float acc = 0.f;
        if (real) {
            const size_t e = ((size_t)token * H + h) * D + sl * 8;
            float a[8], g[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(o + e)), a);
            unpack8(__ldg(reinterpret_cast<const uint4*>(dout + e)), g);
#pragma unroll
            for (int k = 0; k < 8; ++k) acc = fmaf(a[k], g[k], acc);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (valid_row) {
            float* qa = dq_acc + (size_t)r * D + sl * 8;
            reinterpret_cast<float4*>(qa)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            reinterpret_cast<float4*>(qa)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (sl == 0) {
                float l2 = INFINITY;
                if (real) {
                    const float L = cu ? lse[(size_t)h * total + token]
                                       : lse[((size_t)b * H + h) * max_seqlen + pos];
                    l2 = (L == -INFINITY) ? INFINITY : L * 1.4426950408889634f;
                }
                lse2[r] = l2;
                dvec[r] = real ? acc : 0.f;
            }
        }
    }
}

// Deterministic packed conversion: dQ[token, h, :] = scale * the sum, in order
// a = 0, 1, ..., of the accumulators a whose turn count for the row's quarter
// of its tile is nonzero; accumulator rows (h * batch + b) * MSp + pos.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_det_varlen_kernel(const float* __restrict__ acc,
                                                                const int* __restrict__ turn,
                                                                const int* __restrict__ cu,
                                                                __nv_bfloat16* __restrict__ dq, float scale, int H,
                                                                int batch, int max_seqlen, int MSp, int nacc) {
    constexpr int G = D / 8, BR = (D == 128) ? 64 : 128, kMaxAcc = 8;
    const int nqb = MSp / BR;
    const long total = (long)H * batch * MSp * G;
    const size_t acc_elems = (size_t)H * batch * MSp * D, turn_stride = (size_t)H * batch * nqb * 4;
    for (long g = (long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (long)gridDim.x * blockDim.x) {
        const long r = g / G;
        const int c = (int)(g - r * G) * 8;
        const long hb = r / MSp;
        const int pos = (int)(r - hb * MSp);
        const int h = (int)(hb / batch), b = (int)(hb - (long)h * batch);
        if (pos >= varlen_len(cu, b, max_seqlen)) continue;
        const long token = varlen_token(cu, b, max_seqlen, pos);
        const int quarter = (D == 128) ? c / 32 : (pos % 128) / 32;
        const size_t tix = ((size_t)hb * nqb + pos / BR) * 4 + quarter;
        const size_t off = (size_t)r * D + c;
        bool has[kMaxAcc];
#pragma unroll
        for (int a = 0; a < kMaxAcc; ++a) has[a] = a < nacc && __ldg(turn + a * turn_stride + tix) != 0;
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < kMaxAcc; ++a) {
            if (has[a]) {
                const float4* src = reinterpret_cast<const float4*>(acc + a * acc_elems + off);
                const float4 x = __ldg(src), y = __ldg(src + 1);
                s[0] += x.x; s[1] += x.y; s[2] += x.z; s[3] += x.w;
                s[4] += y.x; s[5] += y.y; s[6] += y.z; s[7] += y.w;
            }
        }
        *reinterpret_cast<uint4*>(dq + ((size_t)token * H + h) * D + c) =
            make_uint4(pack_bf16x2(s[0] * scale, s[1] * scale), pack_bf16x2(s[2] * scale, s[3] * scale),
                       pack_bf16x2(s[4] * scale, s[5] * scale), pack_bf16x2(s[6] * scale, s[7] * scale));
    }
}

// dQ[token, h, :] = scale * dQ_acc[(h * batch + b) * MSp + pos, :] for the real rows.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_varlen_kernel(const float* __restrict__ acc, const int* __restrict__ cu,
                                                            __nv_bfloat16* __restrict__ dq, float scale, int H,
                                                            int batch, int max_seqlen, int MSp) {
    constexpr int G = D / 8;  // 8-element groups per row
    const long total = (long)H * batch * MSp * G;
    for (long g = (long)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (long)gridDim.x * blockDim.x) {
        const long r = g / G;
        const int c = (int)(g - r * G) * 8;
        const long hb = r / MSp;
        const int pos = (int)(r - hb * MSp);
        const int h = (int)(hb / batch), b = (int)(hb - (long)h * batch);
        if (pos >= varlen_len(cu, b, max_seqlen)) continue;
        const long token = varlen_token(cu, b, max_seqlen, pos);
        const float4* src = reinterpret_cast<const float4*>(acc + (size_t)r * D + c);
        const float4 x = __ldg(src), y = __ldg(src + 1);
        *reinterpret_cast<uint4*>(dq + ((size_t)token * H + h) * D + c) =
            make_uint4(pack_bf16x2(x.x * scale, x.y * scale), pack_bf16x2(x.z * scale, x.w * scale),
                       pack_bf16x2(y.x * scale, y.y * scale), pack_bf16x2(y.z * scale, y.w * scale));
    }
}

// x / s correctly rounded (IEEE float32 division) for a divisor shared by
// many dividends, by Markstein's method (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with r = 1/s correctly rounded and q = RN(x r), the
// residual x - q s is exact under a fused multiply-add and RN(q + (x - q s) r)
// is the correctly rounded quotient.  Valid while s, 1/s and the quotients
// stay normal; callers use it for 2^-100 < s < 2^100 (quotients below the
// normal range are far below the smallest E4M3 step and quantise to 0 either
// way) and take __fdiv_rn otherwise.  Two dividends at a time: q = RN(x r),
// the residual RN(x - q s) (exact) and RN(q + residual r), each as one
// two-lane instruction.
struct SharedDivisor {
    float s, r;
    __device__ __forceinline__ float2 div2(float2 x) const {
        const float2 q = fmul2(x, make_float2(r, r));
        const float2 res = ffma2(q, make_float2(-s, -s), x);
        return ffma2(res, make_float2(r, r), q);
    }
};

__device__ __forceinline__ SharedDivisor shared_divisor(float s) {
    SharedDivisor d;
    d.s = s;
    d.r = __frcp_rn(s);
    return d;
}

__device__ __forceinline__ bool shared_divisor_ok(float s) { return s > 0x1p-100f && s < 0x1p100f; }

// One CTA iteration (256 threads) per (head, 64-row block); d = 128 -> 8192
// elements, 32 per thread, read once and kept in registers across the
// block's absmax reduction.  The loads of the CTA's next block are issued
// before the current block is reduced and written, so each thread keeps two
// blocks' worth of reads in flight.  s = amax / 448 and x / s are IEEE
// float32 divisions (x / s by SharedDivisor, which gives the same quotients);
// the conversion rounds to nearest even and saturates to +-448.
// The blocks of up to three tensors in one launch (Q, K, V): tensor t has
// rows[t] = B * heads_t heads of N rows each.
struct QuantBlock {
    const __nv_bfloat16* x;
    uint8_t* x8;
    float* scale;
    size_t base;  // first element of the block
    int ng;       // 8-element groups in the block
};

__device__ __forceinline__ QuantBlock quant_block(const QuantJobs& jobs, long gblk, long n0, long n1, int N, int D,
                                                  int nblk) {
    const int t = gblk < n0 ? 0 : gblk < n1 ? 1 : 2;
    const long blk = gblk - (t == 0 ? 0 : t == 1 ? n0 : n1);
    const long bh = blk / nblk;
    const int r0 = (int)(blk - bh * nblk) * 64;
    // selects, not indexing: the parameter arrays stay in the constant bank
    QuantBlock b;
    b.x = reinterpret_cast<const __nv_bfloat16*>(t == 0 ? jobs.x[0] : t == 1 ? jobs.x[1] : jobs.x[2]);
    b.x8 = reinterpret_cast<uint8_t*>(t == 0 ? jobs.x8[0] : t == 1 ? jobs.x8[1] : jobs.x8[2]);
    b.scale = (t == 0 ? jobs.scales[0] : t == 1 ? jobs.scales[1] : jobs.scales[2]) + blk;
    b.base = ((size_t)bh * N + r0) * D;
    b.ng = min(64, N - r0) * (D / 8);
    return b;
}

__global__ void __launch_bounds__(256, 4) quantize_fp8_kernel(const __grid_constant__ QuantJobs jobs, int N, int D, int nblk) {
    constexpr int G = 4;  // uint4 groups (8 elements) per thread: 256 * 4 * 8 = 64 rows x 128
    __shared__ float red[2][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long n0 = (long)jobs.heads[0] * nblk, n1 = n0 + (long)jobs.heads[1] * nblk;
    const long total = n1 + (long)jobs.heads[2] * nblk;
    auto load = [&](const QuantBlock& b, uint4 (&raw)[G]) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int g = threadIdx.x + i * 256;
            raw[i] = (g < b.ng) ? __ldg(reinterpret_cast<const uint4*>(b.x + b.base) + g) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    long gblk = blockIdx.x;
    if (gblk >= total) return;
    QuantBlock nb = quant_block(jobs, gblk, n0, n1, N, D, nblk);
    uint4 nraw[G];
    load(nb, nraw);
    int par = 0;
    for (; gblk < total; gblk += gridDim.x, par ^= 1) {
        const QuantBlock b = nb;
        uint4 raw[G];
#pragma unroll
        for (int i = 0; i < G; ++i) raw[i] = nraw[i];
        if (gblk + gridDim.x < total) {  // the next block's reads go out now
            nb = quant_block(jobs, gblk + gridDim.x, n0, n1, N, D, nblk);
            load(nb, nraw);
        }
        // absmax on the bf16 pairs (exact: a maximum of bf16 values is one of them)
        __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) m2 = __hmax2(m2, __habs2(h[k]));
        }
        float amax = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) red[par][warp] = amax;  // double-buffered: no second barrier per block
        __syncthreads();
        float m = red[par][0];
#pragma unroll
        for (int w = 1; w < 8; ++w) m = fmaxf(m, red[par][w]);
        const float s = (m > 0.f) ? __fdiv_rn(m, 448.f) : 1.f;
        if (threadIdx.x == 0) *b.scale = s;
        float f[G][8];
#pragma unroll
        for (int i = 0; i < G; ++i) unpack8(raw[i], f[i]);
        if (shared_divisor_ok(s)) {  // uniform over the CTA
            const SharedDivisor dv = shared_divisor(s);
#pragma unroll
            for (int i = 0; i < G; ++i)
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    const float2 q = dv.div2(make_float2(f[i][k], f[i][k + 1]));
                    f[i][k] = q.x;
                    f[i][k + 1] = q.y;
                }
        } else {
#pragma unroll
            for (int i = 0; i < G; ++i)
#pragma unroll
                for (int k = 0; k < 8; ++k) f[i][k] = __fdiv_rn(f[i][k], s);
        }
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int g = threadIdx.x + i * 256;
            if (g >= b.ng) continue;
            uint2 out;
            out.x = pack_e4m3x4(f[i][0], f[i][1], f[i][2], f[i][3]);
            out.y = pack_e4m3x4(f[i][4], f[i][5], f[i][6], f[i][7]);
            reinterpret_cast<uint2*>(b.x8 + b.base)[g] = out;
        }
    }
}

__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ y,
                                                          size_t n8) {
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < n8; g += (size_t)gridDim.x * blockDim.x) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(x) + 2 * g);
        const float4 b = __ldg(reinterpret_cast<const float4*>(x) + 2 * g + 1);
        reinterpret_cast<uint4*>(y)[g] =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): the pair carries ~16
// significant bits, enough for float32-accurate scores from bf16 products.
__global__ void __launch_bounds__(256) f32_split_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ hi,
                                                        __nv_bfloat16* __restrict__ lo, size_t n8) {
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < n8; g += (size_t)gridDim.x * blockDim.x) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(x) + 2 * g);
        const float4 b = __ldg(reinterpret_cast<const float4*>(x) + 2 * g + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float h[8], l[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
            l[i] = v[i] - h[i];
        }
        reinterpret_cast<uint4*>(hi)[g] =
            make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
        reinterpret_cast<uint4*>(lo)[g] =
            make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]), pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
    }
}

// Split-key merge.  Partial t of a row holds O_t = (sum over its key range of
// p v) / l_t and LSE_t = m_t + log l_t.  With M = max_t LSE_t,
//   LSE = M + log sum_t exp(LSE_t - M),  O = sum_t exp(LSE_t - LSE) O_t,
// which is the chapter's merge sum_t e^(m_t - m) O~_t / sum_t e^(m_t - m) l_t
// (O~_t the unnormalised partial) rewritten with l_t e^(m_t) = e^(LSE_t).
// All partials -inf (no visible key): O = 0, LSE = -inf.  One warp per row,
// each lane D/32 consecutive head-dim values.
template <int D>
__global__ void lse_merge_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int num_whole,
                                 int num_tail, int S, bool causal, int BH, int num_qp, int N,
                                 __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
    constexpr int V = D / 32;  // values per lane
    const int lane = threadIdx.x & 31;
    const long long nrows = (long long)num_tail * 256;
    for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < nrows;
         r += ((long long)gridDim.x * blockDim.x) >> 5) {
        const int ti = (int)(r >> 8), rr = (int)(r & 255);
        int bh, qp;
        fwd_item_coords(num_whole + ti, causal, BH, num_qp, bh, qp);
        const int row = qp * 256 + rr;
        if (row >= N) continue;
        const size_t base = (size_t)ti * S * 256 + rr;  // partial (ti, 0) of this row
        float M = -INFINITY;
        for (int t = 0; t < S; ++t) M = fmaxf(M, __ldg(lse_part + base + (size_t)t * 256));
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        float out_lse = -INFINITY;
        if (M != -INFINITY) {
            float sw = 0.f;
            for (int t = 0; t < S; ++t) sw += expf(__ldg(lse_part + base + (size_t)t * 256) - M);
            out_lse = M + logf(sw);
            for (int t = 0; t < S; ++t) {
                const float w = expf(__ldg(lse_part + base + (size_t)t * 256) - out_lse);
                const float* src = o_part + (base + (size_t)t * 256) * D + lane * V;
                if constexpr (V == 4) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(src));
                    acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
                } else {
                    const float2 x = __ldg(reinterpret_cast<const float2*>(src));
                    acc[0] += w * x.x; acc[1] += w * x.y;
                }
            }
        }
        const size_t orow = (size_t)bh * N + row;
        __nv_bfloat16* dst = o + orow * D + lane * V;
        if constexpr (V == 4) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
        }
        if (lane == 0) lse[orow] = out_lse;
    }
}

// One warp waits on an mbarrier that nothing ever arrives on, through the same
// bounded wait every pipeline uses; it must give up after `limit_us`, record
// the error bit and return (no trap, no hang).
__global__ void wait_selftest_kernel(unsigned int* err, unsigned long long limit_ns, int* waited_out) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = wait_bounded_warp(smem_u32(&bar), 0, &abort_flag, err, kErrWaitSelftest, limit_ns);
    if (threadIdx.x == 0) *waited_out = ok ? 1 : 0;
}

}  // namespace

// dv[e], dk[e] = sum over s of the split group's partial slices
// part[s][0 (dV) / 1 (dK)][e] (float32, dK already scaled), as bf16.
__global__ void __launch_bounds__(256) dkv_sum_kernel(const float* __restrict__ part, int gsplit, size_t n,
                                                      __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv) {
    const size_t n8 = n / 8;
    for (size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x; g < 2 * n8; g += (size_t)gridDim.x * blockDim.x) {
        const int which = g >= n8;  // 0: dV, 1: dK
        const size_t e = (g - which * n8) * 8;
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int sidx = 0; sidx < gsplit; ++sidx) {
            const float4* src = reinterpret_cast<const float4*>(part + ((size_t)(sidx * 2 + which)) * n + e);
            const float4 x = __ldg(src), y = __ldg(src + 1);
            a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
            a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
        }
        *reinterpret_cast<uint4*>((which ? dk : dv) + e) =
            make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
    }
}

// Block-sparse lists transposed: for every key block k, the query blocks i
// whose list holds k, ascending in i (one CTA, one thread per key block).
// Membership is decided by one binary search per (i, k) in both passes, so
// the counts and the entries written agree even for lists that are not
// ascending; entries outside [0, nkb) are ignored.
__device__ __forceinline__ bool list_holds(const int* __restrict__ col_idx, int a, int e, int k) {
    while (a < e) {
        const int mid = (a + e) >> 1;
        const int v = __ldg(col_idx + mid);
        if (v == k) return true;
        if (v < k) a = mid + 1;
        else e = mid;
    }
    return false;
}

__global__ void __launch_bounds__(1024) block_lists_transpose_kernel(const int* __restrict__ row_ptr,
                                                                     const int* __restrict__ col_idx, int nqb, int nkb,
                                                                     int* __restrict__ col_ptr,
                                                                     int* __restrict__ row_idx) {
    extern __shared__ int cnt[];  // [nkb + 1]
    const int nnz = __ldg(row_ptr + nqb);
    for (int k = threadIdx.x; k < nkb; k += blockDim.x) {
        int c = 0;
        for (int i = 0; i < nqb; ++i) {
            const int a = min(max(__ldg(row_ptr + i), 0), nnz), e = min(max(__ldg(row_ptr + i + 1), a), nnz);
            c += list_holds(col_idx, a, e, k);
        }
        cnt[k] = c;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int k = 0; k < nkb; ++k) {
            const int c = cnt[k];
            cnt[k] = run;
            col_ptr[k] = run;
            run += c;
        }
        col_ptr[nkb] = run;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < nkb; k += blockDim.x) {
        int pos = cnt[k];
        for (int i = 0; i < nqb; ++i) {
            const int a = min(max(__ldg(row_ptr + i), 0), nnz), e = min(max(__ldg(row_ptr + i + 1), a), nnz);
            if (list_holds(col_idx, a, e, k)) row_idx[pos++] = i;
        }
    }
}

cudaError_t launch_lse_merge(const float* o_part, const float* lse_part, int num_whole, int num_tail, int splits,
                             bool causal, int BH, int num_qp, int N, int d, void* o, float* lse, cudaStream_t stream) {
    if (num_tail <= 0 || splits <= 1) return cudaSuccess;
    const long long blocks = ((long long)num_tail * 256 + 7) / 8;  // 8 rows (warps) per block
    const int grid = (int)(blocks < 152 * 32 ? blocks : 152 * 32);
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(o);
    if (d == 128)
        lse_merge_kernel<128><<<grid, 256, 0, stream>>>(o_part, lse_part, num_whole, num_tail, splits, causal, BH,
                                                        num_qp, N, ob, lse);
    else
        lse_merge_kernel<64><<<grid, 256, 0, stream>>>(o_part, lse_part, num_whole, num_tail, splits, causal, BH,
                                                       num_qp, N, ob, lse);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre_varlen(const void* o, const void* dout, const float* lse, const int* cu, float* lse2,
                                  float* dvec, float* dq_acc, int H, int batch, int total, int max_seqlen, int MSp,
                                  int d, int grid, cudaStream_t s) {
    const __nv_bfloat16* ob = reinterpret_cast<const __nv_bfloat16*>(o);
    const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(dout);
    if (d == 128)
        bwd_pre_varlen_kernel<128><<<grid, 256, 0, s>>>(ob, gb, lse, cu, lse2, dvec, dq_acc, H, batch, total,
                                                        max_seqlen, MSp);
    else
        bwd_pre_varlen_kernel<64><<<grid, 256, 0, s>>>(ob, gb, lse, cu, lse2, dvec, dq_acc, H, batch, total,
                                                       max_seqlen, MSp);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_varlen(const float* acc, const int* cu, void* dq, float scale, int H, int batch,
                                 int max_seqlen, int MSp, int d, int grid, cudaStream_t s) {
    __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(dq);
    if (d == 128)
        bwd_dq_varlen_kernel<128><<<grid, 256, 0, s>>>(acc, cu, q, scale, H, batch, max_seqlen, MSp);
    else
        bwd_dq_varlen_kernel<64><<<grid, 256, 0, s>>>(acc, cu, q, scale, H, batch, max_seqlen, MSp);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned int* err, unsigned int limit_us, int* waited_out, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, (unsigned long long)limit_us * 1000ull, waited_out);
    return cudaGetLastError();
}

cudaError_t launch_f32_split_bf16(const float* x, void* hi, void* lo, size_t n, int grid, cudaStream_t s) {
    f32_split_kernel<<<grid, 256, 0, s>>>(x, reinterpret_cast<__nv_bfloat16*>(hi), reinterpret_cast<__nv_bfloat16*>(lo),
                                          n / 8);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const void* o, const void* dout, bool in_f32, const float* lse, float* lse2, float* dvec,
                           float* dq_acc, int BH, int N, int Np, int d, int grid, cudaStream_t s) {
    if (d == 128) {
        if (in_f32) bwd_pre_kernel<128, true><<<grid, 256, 0, s>>>(o, dout, lse, lse2, dvec, dq_acc, BH, N, Np);
        else bwd_pre_kernel<128, false><<<grid, 256, 0, s>>>(o, dout, lse, lse2, dvec, dq_acc, BH, N, Np);
    } else {
        if (in_f32) bwd_pre_kernel<64, true><<<grid, 256, 0, s>>>(o, dout, lse, lse2, dvec, dq_acc, BH, N, Np);
        else bwd_pre_kernel<64, false><<<grid, 256, 0, s>>>(o, dout, lse, lse2, dvec, dq_acc, BH, N, Np);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_det_varlen(const float* acc, const int* turn, const int* cu_seqlens, void* dq, float scale,
                                     int H, int batch, int max_seqlen, int MSp, int d, int nacc, int grid,
                                     cudaStream_t s) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(dq);
    if (d == 128)
        bwd_dq_det_varlen_kernel<128><<<grid, 256, 0, s>>>(acc, turn, cu_seqlens, o, scale, H, batch, max_seqlen, MSp,
                                                           nacc);
    else
        bwd_dq_det_varlen_kernel<64><<<grid, 256, 0, s>>>(acc, turn, cu_seqlens, o, scale, H, batch, max_seqlen, MSp,
                                                          nacc);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_det(const float* acc, const int* turn, void* dq, float scale, int BH, int N, int Np, int d,
                              int nacc, int grid, cudaStream_t s) {
    bwd_dq_det_kernel<<<grid, 256, 0, s>>>(acc, turn, reinterpret_cast<__nv_bfloat16*>(dq), scale, BH, N, Np, d, nacc);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre_fp8(const void* o, const void* do8, const float* sdo, const float* lse, float* lse2,
                               float* dvec, float* dq_acc, int BH, int N, int Np, int grid, cudaStream_t s) {
    bwd_pre_fp8_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(o),
                                            reinterpret_cast<const uint8_t*>(do8), sdo, lse, lse2, dvec, dq_acc, BH,
                                            N, Np, (N + 63) / 64);
    return cudaGetLastError();
}

// CTAs that fit on the GPU at once (256 threads each), for the grid-stride
// kernels whose grid should not spill into a partial second wave.
template <class K>
int resident_ctas(K kernel, int sms) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 1;
    }
    return sms * (n > 0 ? n : 1);
}

cudaError_t launch_bwd_dq(const float* dq_acc, void* dq, bool out_f32, float scale, int BH, int N, int Np, int d,
                          int sms, cudaStream_t s) {
    static const int per_f32 = resident_ctas(bwd_dq_kernel<true>, 1), per_bf16 = resident_ctas(bwd_dq_kernel<false>, 1);
    if (out_f32) bwd_dq_kernel<true><<<sms * per_f32, 256, 0, s>>>(dq_acc, dq, scale, BH, N, Np, d);
    else bwd_dq_kernel<false><<<sms * per_bf16, 256, 0, s>>>(dq_acc, dq, scale, BH, N, Np, d);
    return cudaGetLastError();
}

cudaError_t launch_dkv_sum(const float* part, int gsplit, size_t n, void* dk, void* dv, int grid, cudaStream_t s) {
    dkv_sum_kernel<<<grid, 256, 0, s>>>(part, gsplit, n, reinterpret_cast<__nv_bfloat16*>(dk),
                                        reinterpret_cast<__nv_bfloat16*>(dv));
    return cudaGetLastError();
}

cudaError_t launch_block_lists_transpose(const int* row_ptr, const int* col_idx, int nqb, int nkb, int* col_ptr,
                                         int* row_idx, cudaStream_t s) {
    const int threads = nkb < 1024 ? ((nkb + 31) / 32) * 32 : 1024;
    block_lists_transpose_kernel<<<1, threads, (nkb + 1) * sizeof(int), s>>>(row_ptr, col_idx, nqb, nkb, col_ptr,
                                                                             row_idx);
    return cudaGetLastError();
}

// Test hook: q[i] = x[i] / s[i % ns] by SharedDivisor and by __fdiv_rn.
__global__ void shared_div_check_kernel(const float* __restrict__ x, const float* __restrict__ s, int ns, size_t n,
                                        float* __restrict__ q_fast, float* __restrict__ q_ieee) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float d = s[i % ns];
        // the pair form the quantiser uses, its lanes taken in turn
        const float2 q = shared_divisor(d).div2(make_float2(x[i], x[i]));
        q_fast[i] = (i & 1) ? q.y : q.x;
        q_ieee[i] = __fdiv_rn(x[i], d);
    }
}

cudaError_t launch_shared_div_check(const float* x, const float* s, int ns, size_t n, float* q_fast, float* q_ieee,
                                    cudaStream_t st) {
    shared_div_check_kernel<<<1024, 256, 0, st>>>(x, s, ns, n, q_fast, q_ieee);
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const QuantJobs& jobs, int N, int d, int sms, cudaStream_t s) {
    const int nblk = (N + 63) / 64;
    // The CTAs loop over the blocks, so the grid is what fits on the GPU at
    // once: a larger grid would run as a partial second wave, each late CTA
    // taking its share of blocks after the others have finished.
    static const int per_sm = resident_ctas(quantize_fp8_kernel, 1);
    const long long blocks = (long long)(jobs.heads[0] + jobs.heads[1] + jobs.heads[2]) * nblk;
    const int grid = (int)std::min<long long>(blocks, (long long)sms * per_sm);
    if (grid <= 0) return cudaSuccess;
    quantize_fp8_kernel<<<grid, 256, 0, s>>>(jobs, N, d, nblk);
    return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* x, void* y, size_t n, int grid, cudaStream_t s) {
    f32_to_bf16_kernel<<<grid, 256, 0, s>>>(x, reinterpret_cast<__nv_bfloat16*>(y), n / 8);
    return cudaGetLastError();
}

}  // namespace fa

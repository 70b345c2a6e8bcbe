// Shared definitions of the device code: kernel parameter blocks, device error
// codes and the launch entry points the C ABI layer calls.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "checks.h"

namespace fa {

// Bits of the device error word (set by a kernel whose pipeline wait timed out).
enum : unsigned int {
    kErrWaitFwdProducer = 1u << 0,
    kErrWaitFwdMma = 1u << 1,
    kErrWaitFwdSoftmax = 1u << 2,
    kErrWaitBwdProducer = 1u << 3,
    kErrWaitBwdMma = 1u << 4,
    kErrWaitBwdCompute = 1u << 5,
    kErrWaitBwdDq = 1u << 6,
    kErrWaitDrain = 1u << 7,
    kErrWaitSelftest = 1u << 8,
    kErrWaitBwdDqTurn = 1u << 9,
};

constexpr int kNumSMsDefault = 152;

// Work order of the persistent kernels.  Items are numbered longest first
// (causal: the query tiles, resp. key blocks, that see the most keys, resp.
// queries); a CTA takes one item per round of gridDim.x items, and the rounds
// alternate direction ("snake": CTA c takes rank r*G + c in even rounds and
// r*G + G-1-c in odd ones), so that a CTA given a long item in one round gets
// a short one in the next and the per-CTA totals stay near the mean.  Returns
// -1 for a round in which this CTA has no item (the last, partial round).
__device__ __forceinline__ int snake_item(int round, int num_items) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const int it = round * G + ((round & 1) ? (G - 1 - c) : c);
    return it < num_items ? it : -1;
}
__device__ __forceinline__ int snake_rounds(int num_items) { return (num_items + (int)gridDim.x - 1) / (int)gridDim.x; }

// Forward work item `it` (longest first) -> (head index bh, query-row pair qp).
__host__ __device__ __forceinline__ void fwd_item_coords(int it, bool causal, int BH, int num_qp, int& bh, int& qp) {
    if (causal) {  // the pairs that see the most keys first
        qp = num_qp - 1 - it / BH;
        bh = it % BH;
    } else {
        qp = it % num_qp;
        bh = it / num_qp;
    }
}

struct FwdParams {
    int B, H, N;
    int Hkv;          // key/value heads (H % Hkv == 0): query head h reads key/value head h / (H / Hkv)
    int num_qp;       // query-row pairs of 128-row tiles per head: ceil(N / 256)
    int num_items;    // B * H * num_qp
    // Split keys (FlashDecoding form): work units 0 .. num_whole-1 are whole
    // items; each later item is cut into `splits` contiguous key ranges, one
    // unit each, whose normalised O and LSE go to o_part / lse_part (unit
    // u >= num_whole is partial u - num_whole) for the merge kernel.
    int num_units;    // num_whole + (num_items - num_whole) * splits
    int num_whole;
    int splits;
    float* o_part;    // [partials][256 rows][d] f32
    float* lse_part;  // [partials][256 rows]
    float scale;      // softmax scale applied to Q K^T
    float scale_log2; // scale * log2(e)
    // Packed variable-length sequences (VARLEN instance): sequence b holds
    // tokens cu_seqlens[b] .. cu_seqlens[b+1]-1; q, o are [total, H, d], k, v
    // [total, Hkv, d], lse [H, total]; B is the number of sequences and N the
    // longest length.  They share storage with fields that instance does not
    // read, so that the struct keeps its size: a larger parameter block had
    // slowed the other forward instances by several percent.
    union {
        const int* kv_lens;     // [B] valid keys per batch item, or NULL
        const int* cu_seqlens;  // [B + 1] (VARLEN)
    };
    void* o;          // [B,H,N,d] bf16 or f32
    float* lse;       // [B,H,N]
    const float* sq;  // FP8 only: per-64-row-block scales [B,H,nblk]
    union {
        const float* sk;
        const int* cu_seqlens_k;  // VARLEN: [B + 1] key token ranges, or NULL (= cu_seqlens)
    };
    const float* sv;
    union {
        int nblk;     // ceil(N / 64) (FP8)
        int total;    // packed tokens (VARLEN)
    };
    unsigned int* err;
};

struct BwdParams {
    int B, H, N, Np;  // Np: N padded to a multiple of 128
    int Hkv;          // key/value heads (H % Hkv == 0); dK, dV are [B,Hkv,N,d]
    int num_kt;       // key tiles per head: ceil(N / 128)
    int num_items;    // B * Hkv * num_kt
    float scale;
    float scale_log2;
    union {
        const int* kv_lens;
        const int* cu_seqlens_k;  // packed: [B + 1] key token ranges, or NULL (= cu_seqlens)
    };
    const float* lse2;  // [B,H,Np] LSE * log2(e), +inf on rows with no visible key / padding
    const float* dvec;  // [B,H,Np] D = rowsum(dO * O)
    float* dq_acc;      // [B,H,Np,d] float32 accumulator (unscaled)
    void* dk;           // [B,Hkv,N,d]
    void* dv;
    // packed variable-length sequences (see FwdParams): B sequences, N the
    // longest; statistics and dQ accumulator rows (h * B + b) * Np + position
    const int* cu_seqlens;
    int total;
    unsigned int* err;
    // Shared key/value heads with few key blocks: each key block's group of
    // query heads is split over gsplit work units; unit s writes float32
    // partial dV, scale * dK to dkv_part [gsplit][2 (dV, dK)][B*Hkv][N][d],
    // summed into dv, dk by a separate kernel.  gsplit = 1: written directly.
    int gsplit;
    float* dkv_part;
};

// Sliding window (flash_attn_func's window_size, chapter 18 §18.7.1): key j
// is visible to query i only if i - win_left <= j <= i + win_right, -1
// meaning no bound on that side.  Derived types, so that only the window
// instances carry the two fields.
struct FwdParamsWin : FwdParams {
    int win_left, win_right;
};
struct BwdParamsWin : BwdParams {
    int win_left, win_right;
};

// Rectangular attention (decoding against a key/value cache, cross-attention):
// Nk keys (K, V have Nk rows).  The query rows of the g heads sharing a
// key/value head are contiguous in [B, H, Nq, d], so they are packed as the
// N = g * Nq rows of one "head" (H here is the number of key/value heads):
// row r is query r % qmod (qmod = Nq) of its head, and with the causal mask
// it sees keys j <= r % qmod + coff, coff = Nk - Nq.
struct FwdParamsRect : FwdParams {
    int Nk, coff, qmod;
};

// Block-sparse attention (chapter 18 §18.8.1): the 128-row query block i
// computes only the 128-key blocks col_idx[row_ptr[i] .. row_ptr[i+1]-1]
// (ascending), one list for every batch item and head.  The backward reads
// the transposed lists (per key block, its query blocks, ascending), which
// the library builds in the workspace.
struct FwdParamsSparse : FwdParams {
    const int* row_ptr;  // [nqb + 1]
    const int* col_idx;  // [row_ptr[nqb]]
    int nqb, nkb;
};
// Rectangular backward: N query rows (statistics, dQ), Nk keys (K, V, dK,
// dV); with the causal mask query i sees keys j <= i + coff, coff = Nk - N.
struct BwdParamsRect : BwdParams {
    int Nk, coff;
};
struct BwdParamsSparse : BwdParams {
    const int* col_ptr;  // [nkb + 1]
    const int* row_idx;
    int nqb, nkb;
    const int* row_ptr;  // the forward lists (deterministic instance only)
    const int* col_idx;
};
// Deterministic backward: nacc float32 dQ accumulators [nacc][B*H][Np][d]
// (the first is dq_acc); key block kt writes accumulator kt % nacc, and each
// accumulator tile of (query head row bhq, query block i) receives its key
// blocks in increasing order: the first one stores, the others add.
// dq_turn[((a * B*H + bhq) * nqt + i) * 4 + w] (nqt = Np / query rows per
// step; w = the drain warp's quarter of the tile) counts the contributions to
// quarter w of that tile of accumulator a; key block kt writes once it reaches
// its rank among the key blocks visiting that query block in accumulator a
// (key blocks first(i), first(i) + 1, ... visit query block i: first(i) = 0
// except under a sliding window).  The conversion sums the accumulators with
// a nonzero count in order a = 0, 1, ...  Key blocks that run at the same time
// go to different accumulators, so they seldom wait for one another.  BwdDet
// adds these fields to any of the backward parameter blocks.
template <class Base>
struct BwdDet : Base {
    int* dq_turn;
    int nqt;  // query tiles of BR rows per head row: Np / BR
    int nacc;
};
using BwdParamsDet = BwdDet<BwdParams>;

// FP8 backward (d = 128): E4M3 codes of Q, K, V, dO with one float32 scale
// per 64-row block ([B*H][nblk]); float32 dK, dV [B,H,N,128]; statistics and
// the float32 dQ accumulator as for the bf16 backward.
struct BwdFp8Params {
    int B, H, N, Np, nblk;
    int num_kt, num_items, causal;
    float scale, scale_log2;
    const int* kv_lens;
    const float* sq;
    const float* sk;
    const float* sv;
    const float* sdo;
    const float* lse2;
    const float* dvec;
    float* dk;
    float* dv;
    unsigned int* err;
};

// Launch helpers implemented in the kernel translation units.  They return a
// cudaError_t from the launch itself.
// Tensor maps of one forward launch: q, k, v and, for float32 inputs carried
// as bf16 hi + lo parts, the low parts of q and k.
struct FwdMaps {
    CUtensorMap q, k, v, q_lo, k_lo;
};
cudaError_t launch_fwd_bf16_d64(int block_c, bool causal, bool out_f32, bool split, const FwdMaps& m,
                                const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_bf16_d128(int block_c, bool causal, bool out_f32, bool split, const FwdMaps& m,
                                 const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_window(int d, const FwdMaps& m, const FwdParamsWin& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_rect(int d, bool causal, const FwdMaps& m, const FwdParamsRect& p, int grid,
                            cudaStream_t stream);
cudaError_t launch_fwd_sparse(int d, bool causal, const FwdMaps& m, const FwdParamsSparse& p, int grid,
                              cudaStream_t stream);
cudaError_t launch_bwd_main_sparse(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                   const BwdParamsSparse& p, int grid, cudaStream_t stream);
// Test hook of the quantiser's division: q_fast = x / s by the shared-divisor
// method, q_ieee = __fdiv_rn(x, s), s[i % ns] for element i.
cudaError_t launch_shared_div_check(const float* x, const float* s, int ns, size_t n, float* q_fast, float* q_ieee,
                                    cudaStream_t stream);
// dv, dk = sums of the gsplit partial slices (bf16).
cudaError_t launch_dkv_sum(const float* part, int gsplit, size_t n, void* dk, void* dv, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_rect(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsRect& p, int grid,
                                 cudaStream_t stream);
// Deterministic backward (shared key/value heads allowed; p.dq_turn zeroed),
// and its dQ conversion: dq = scale * the sum of the written accumulators.
cudaError_t launch_bwd_dq_det(const float* acc, const int* turn, void* dq, float scale, int BH, int N, int Np, int d,
                              int nacc, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_det_window(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdDet<BwdParamsWin>& p,
                                       int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_det_rect(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                     const BwdDet<BwdParamsRect>& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_det_sparse(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                       const BwdDet<BwdParamsSparse>& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_varlen_window(int d, const FwdMaps& m, const FwdParamsWin& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_varlen_window(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                          const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsWin& p,
                                          int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_det_varlen_window(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                                              const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                              const BwdDet<BwdParamsWin>& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_det_varlen(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                       const BwdParamsDet& p, int grid, cudaStream_t stream);
// Packed layout ([H][batch][MSp] accumulator rows, token-major dq):
cudaError_t launch_bwd_dq_det_varlen(const float* acc, const int* turn, const int* cu_seqlens, void* dq, float scale,
                                     int H, int batch, int max_seqlen, int MSp, int d, int nacc, int grid,
                                     cudaStream_t stream);
cudaError_t launch_bwd_main_det(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsDet& p, int grid,
                                cudaStream_t stream);
// Transposes the query-block lists into per-key-block lists (one CTA).
cudaError_t launch_block_lists_transpose(const int* row_ptr, const int* col_idx, int nqb, int nkb, int* col_ptr,
                                         int* row_idx, cudaStream_t stream);
cudaError_t launch_bwd_main_window(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParamsWin& p, int grid,
                                   cudaStream_t stream);
cudaError_t launch_fwd_varlen(int d, bool causal, const FwdMaps& m, const FwdParams& p, int grid,
                              cudaStream_t stream);
cudaError_t launch_fwd_splitk(int d, bool fp8, bool causal, const FwdMaps& m, const FwdParams& p, int grid,
                              cudaStream_t stream);
cudaError_t launch_fwd_fp8_d128(bool causal, const FwdMaps& m, const FwdParams& p, int grid,
                                cudaStream_t stream);
cudaError_t launch_bwd_main_varlen(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                   const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main_gqa(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                                const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_main(int d, bool causal, bool out_f32, const CUtensorMap& tq,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdq, const BwdParams& p, int grid,
                            cudaStream_t stream);
// FP8 backward main kernel; tkt: the transposed K codes [B*H][128][Np].
cudaError_t launch_bwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                           const CUtensorMap& tkt, const CUtensorMap& tdq, const BwdFp8Params& p, int grid,
                           cudaStream_t stream);
// FP8 backward preprocess: D = rowsum(s_do dO8 * O), LSE * log2(e), zeroed
// dQ accumulator (d = 128; o bf16, do8 E4M3 codes with per-64-row scales).
cudaError_t launch_bwd_pre_fp8(const void* o, const void* do8, const float* sdo, const float* lse, float* lse2,
                               float* dvec, float* dq_acc, int BH, int N, int Np, int grid, cudaStream_t stream);
// k8 [B*H][N][128] -> kt [B*H][128][Np] (uint8 codes; keys >= N zero).
cudaError_t launch_transpose_k8(const void* k8, void* kt, int BH, int N, int Np, int grid, cudaStream_t stream);
cudaError_t launch_bwd_pre(const void* o, const void* dout, bool in_f32, const float* lse,
                           float* lse2, float* dvec, float* dq_acc, int BH, int N, int Np, int d,
                           int grid, cudaStream_t stream);
cudaError_t launch_bwd_dq(const float* dq_acc, void* dq, bool out_f32, float scale, int BH, int N,
                          int Np, int d, int sms, cudaStream_t stream);
// Up to three tensors quantised by one launch (unused slots: heads = 0).
struct QuantJobs {
    const void* x[3];  // bf16
    void* x8[3];       // E4M3 codes
    float* scales[3];
    int heads[3];  // B * heads of each tensor
};
cudaError_t launch_quantize_fp8(const QuantJobs& jobs, int N, int d, int sms, cudaStream_t stream);
// Merges the split-key partials of the forward into O (bf16) and LSE.
cudaError_t launch_lse_merge(const float* o_part, const float* lse_part, int num_whole, int num_tail, int splits,
                             bool causal, int BH, int num_qp, int N, int d, void* o, float* lse, cudaStream_t stream);
cudaError_t launch_bwd_pre_varlen(const void* o, const void* dout, const float* lse, const int* cu, float* lse2,
                                  float* dvec, float* dq_acc, int H, int batch, int total, int max_seqlen, int MSp,
                                  int d, int grid, cudaStream_t stream);
cudaError_t launch_bwd_dq_varlen(const float* acc, const int* cu, void* dq, float scale, int H, int batch,
                                 int max_seqlen, int MSp, int d, int grid, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned int* err, unsigned int limit_us, int* waited_out,
                                 cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float* x, void* y, size_t n, int grid, cudaStream_t stream);
cudaError_t launch_f32_split_bf16(const float* x, void* hi, void* lo, size_t n, int grid,
                                  cudaStream_t stream);

}  // namespace fa

// Persistent backward kernel of exact tiled attention for sm_103a.
//
// What it computes is Algorithm 2 of the FA-v2 analysis page
// ("解析 FlashAttention（4）：FlashAttention-v2", §5.4), in that page's loop
// order: the outer loop over key/value blocks j is the CTA work item, the inner
// loop walks query blocks i.  Per (i, j):
//   P  = exp(S - L_i)            S = scale Q_i K_j^T (masked), L_i = saved LSE
//   dV_j += P^T dO_i
//   dP = dO_i V_j^T
//   dS = P (dP - D_i)            D_i = rowsum(dO_i O_i), from the preprocess
//   dQ_i += dS K_j               (reduced into a float32 accumulator)
//   dK_j += dS^T Q_i
// with the 1/sqrt(d) factor of the attention-kernels wiki §04 applied to dK in
// the epilogue and to dQ in the conversion kernel.  Rows with LSE = -inf
// (no visible key) carry L*log2(e) = +inf so their P is exactly 0.
//
// GB300 mapping (one CTA per SM, persistent over (head, key block) items):
//   * the key block (128 keys) is the M = 128 side of every MMA, so K_j, V_j
//     stay on chip for the item and dK_j, dV_j accumulate in TMEM;
//   * S^T = K_j Q_i^T and dP^T = V_j dO_i^T land in TMEM with one key per lane;
//     at d = 128 their A operands K_j, V_j are read from TMEM (copied there
//     once per item by warps 8-11), which takes 32 KB of operand reads per
//     step off shared memory and lets those N = 64 products run at their
//     math rate;
//   * two compute warpgroups (warps 0-3, 4-7) each own half of the query
//     columns: P^T goes back to TMEM (bf16, aliased on S^T) as the A operand of
//     dV += P^T dO_i; dS^T is written to shared memory in the 128-byte-swizzle
//     layout, which serves both as the K-major A operand of dK += dS^T Q_i and
//     as the MN-major operand of the dQ product;
//   * d = 128: dQ_i^T = K_j^T dS^T (M = 128 head-dim lanes, N = 64 queries);
//     d = 64:  dQ_i = dS K_j (M = 128 query lanes, N = 64).  Either way all
//     MMAs have M = 128;
//   * TMEM holds one step slot: S^T, and dP^T whose columns are reused for
//     dQ^T once dS is formed (d = 128; d = 64 has a separate dQ region).  The
//     MMA warp issues S of the next step while the compute warpgroups work on
//     the current one, and its dP once the current dQ^T has been drained;
//   * warps 8-11 drain the dQ tile from TMEM into shared memory and add it to
//     the float32 accumulator with asynchronous bulk reductions (TMA), each
//     warp independently; at d = 128 they also copy K_j, V_j into TMEM at
//     the start of each item;
//   * warp 12 issues TMA loads (K_j, V_j once per item; a ring of Q_i, dO_i
//     and the row statistics), warp 13 issues tcgen05.mma.
#pragma once
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kThreads = 448;
constexpr int kDqWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
// Deterministic instance: a drain warp passes a tile's turn on kDetLag steps
// after writing it, when the write has completed, so that it never waits for
// a write in flight.
constexpr int kDetLag = 4;

template <int D_>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int BC = 128;                    // keys per item (TMEM lanes)
    static constexpr int BR = (D == 128) ? 64 : 128;  // queries per inner step
    static constexpr int HALF = BR / 2;               // query columns per compute warpgroup
    static constexpr int NSLOT = 1;                   // TMEM step slots
    // d = 128: K_j and V_j are also copied into TMEM (bf16, two per column) and
    // serve as the A operands of S^T and dP^T, so those products read only
    // their 2 KB of Q_i / dO_i per instruction from shared memory
    static constexpr bool KV_TMEM = (D == 128);
    static constexpr bool DQ_ALIAS = (D == 128);      // dQ reuses the slot's dP columns
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int NBOX = ROW_BYTES / 128;
    static constexpr int K_BOX = BC * 128, K_TILE = BC * ROW_BYTES;
    static constexpr int Q_BOX = BR * 128, Q_TILE = BR * ROW_BYTES;
    static constexpr int DS_BOX = BC * 128, DS_TILE = BC * BR * 2;
    static constexpr int DQ_WARP_BYTES = 8192;        // per drain warp staging
    static constexpr int STAGES = (D == 128) ? 3 : 2;  // Q/dO ring
    // TMEM columns: dV | dK | [K | V] | slot (S, X) | [dQ]
    static constexpr int TM_DV = 0, TM_DK = D;
    static constexpr int TM_K = 2 * D, TM_V = 2 * D + D / 2;  // used when KV_TMEM
    static constexpr int TM_SLOT0 = KV_TMEM ? 3 * D : 2 * D, TM_SLOT = 2 * BR;
    static constexpr int TM_DQ = DQ_ALIAS ? -1 : TM_SLOT0 + NSLOT * TM_SLOT;
    static constexpr int TM_COLS = 512;
    static_assert(TM_SLOT0 + NSLOT * TM_SLOT + (DQ_ALIAS ? 0 : 64) <= TM_COLS, "TMEM budget");
    // shared memory map
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + K_TILE;
    static constexpr int OFF_Q = OFF_V + K_TILE;
    static constexpr int OFF_DO = OFF_Q + STAGES * Q_TILE;
    static constexpr int OFF_DS = OFF_DO + STAGES * Q_TILE;
    static constexpr int OFF_DQ = OFF_DS + 2 * DS_TILE;
    static constexpr int OFF_STAT = OFF_DQ + 4 * DQ_WARP_BYTES;  // per stage: lse2[BR], D[BR]
    static constexpr int STAT_BYTES = 2 * BR * 4;
    static constexpr int OFF_BAR = OFF_STAT + STAGES * STAT_BYTES;
    static constexpr int B_KVFULL = 0, B_KVEMPTY = 1;
    static constexpr int B_QFULL = 2, B_QEMPTY = 2 + STAGES;
    static constexpr int B_SFULL = 2 + 2 * STAGES;  // [NSLOT] each below
    static constexpr int B_DPFULL = B_SFULL + 2, B_PFULL = B_DPFULL + 2, B_DSFULL = B_PFULL + 2;
    static constexpr int B_DSEMPTY = B_DSFULL + 2;  // [2] (dS buffers)
    static constexpr int B_DQFULL = B_DSEMPTY + 2, B_DQEMPTY = B_DQFULL + 2;
    static constexpr int B_ACCFULL = B_DQEMPTY + 2, B_ACCEMPTY = B_ACCFULL + 1;
    static constexpr int B_DONE = B_ACCEMPTY + 1;
    static constexpr int B_KVTFULL = B_DONE + 1;  // K_j, V_j copied into TMEM
    static constexpr int NBAR = B_KVTFULL + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static_assert(SMEM <= 232448, "shared memory budget");
    static constexpr uint32_t IDESC_S = idesc_make(kFmtBF16, kFmtBF16, 0, 0, 128, BR);   // S^T, dP^T
    static constexpr uint32_t IDESC_ACC = idesc_make(kFmtBF16, kFmtBF16, 0, 1, 128, D);  // dV, dK
    static constexpr uint32_t IDESC_DQ = idesc_make(kFmtBF16, kFmtBF16, 1, 1, 128, 64);  // dQ^T / dQ
    __host__ __device__ static constexpr int s_col(int slot) { return TM_SLOT0 + slot * TM_SLOT; }
    __host__ __device__ static constexpr int x_col(int slot) { return TM_SLOT0 + slot * TM_SLOT + BR; }
    __host__ __device__ static constexpr int dq_col(int slot) { return DQ_ALIAS ? x_col(slot) : TM_DQ; }
};

// A work item is one key block of one key/value head: bh = b * Hkv + kv head
// (the K, V, dK, dV row).  Its steps run over the query heads sharing that
// key/value head (qh0 .. qh0 + H/Hkv - 1; one head without sharing) and, for
// each, the query blocks i0 .. i0 + ni - 1, so dK and dV sum over the group.
struct Item {
    int bh, b, kt, kvl, i0, n;
    int qh0, ni;  // first query head row (b * H + ...), query blocks per query head
    int kvh, tb, seqlen;  // packed sequences: key/value head in the sequence, first token, length
    int tbk, coff;        // packed: first key token, causal offset (keys - queries) of the sequence
    int sub;              // split group: which part of the query heads (0 .. gsplit - 1)
};

// GQA: the kernel instance for shared key/value heads (compiled separately so
// that the plain backward carries none of the group bookkeeping).
// VARLEN (packed variable-length sequences, always with the GQA step loop):
// qh0 / the step's bhq are head indices within the sequence, the K, V, dK, dV
// rows are tokens tb + key, and the statistics rows are (h * B + b) * Np + ...
// WINDOW: the sliding-window instance (p is a BwdParamsWin; causal is folded
// into the window's right edge by the caller).
// SPARSE: the block-sparse instance (p is a BwdParamsSparse): key block kt
// visits the 128-row query blocks row_idx[i0 .. i0 + ni / R - 1] (R steps
// per query block), per query head of its group.
// RECT: the rectangular instance (p is a BwdParamsRect): N query rows, Nk keys.
template <bool WINDOW, bool SPARSE = false, bool RECT = false>
using ParamsT = typename std::conditional<
    WINDOW, BwdParamsWin,
    typename std::conditional<SPARSE, BwdParamsSparse,
                              typename std::conditional<RECT, BwdParamsRect, BwdParams>::type>::type>::type;

// DET: the deterministic instance (p is a BwdDet<...>; all but block-sparse):
// each drain warp adds its quarter of a dQ tile only on its turn.
template <bool WINDOW, bool SPARSE, bool RECT, bool DET>
using KernelParamsT =
    typename std::conditional<DET, BwdDet<ParamsT<WINDOW, SPARSE, RECT>>, ParamsT<WINDOW, SPARSE, RECT>>::type;

// Keys of a head (K, V, dK, dV rows) and the causal offset.
template <class PT>
__device__ __forceinline__ int key_count(const PT& p) {
    if constexpr (std::is_base_of<BwdParamsRect, PT>::value) return p.Nk;
    else return p.N;
}
template <class PT>
__device__ __forceinline__ int causal_offset(const PT& p) {
    if constexpr (std::is_base_of<BwdParamsRect, PT>::value) return p.coff;
    else return 0;
}

template <class C, bool CAUSAL, bool GQA, bool VARLEN = false, bool WINDOW = false, bool SPARSE = false,
          bool RECT = false, bool DET = false>
__device__ __forceinline__ Item get_item(int it, const ParamsT<WINDOW, SPARSE, RECT>& p) {
    Item I;
    const int Hkv = GQA ? p.Hkv : p.H;
    const int BH = p.B * Hkv;
    // split group (GQA, not packed): consecutive units share a key block
    const int gs = (GQA && !VARLEN) ? max(p.gsplit, 1) : 1;
    I.sub = 0;
    if (gs > 1) {
        I.sub = it % gs;
        it /= gs;
    }
    // causal: key blocks near the start see the most query rows: first.
    // DET: key block major too, so that the key blocks of a head running at
    // the same time are few and consecutive (they use different accumulators)
    if (CAUSAL || DET) {
        I.kt = it / BH;
        I.bh = it % BH;
    } else {
        I.bh = it / p.num_kt;
        I.kt = it % p.num_kt;
    }
    dcheck(chk::tile_ok(I.bh, BH, I.kt, p.num_kt), kErrCheckTile);
    I.b = I.bh / Hkv;
    const int group = GQA ? p.H / Hkv : 1;
    const int gper = group / gs;  // query heads of this unit
    I.kvh = I.bh - I.b * Hkv;
    I.qh0 = VARLEN ? I.kvh * group : GQA ? I.b * p.H + I.kvh * group + I.sub * gper : I.bh;
    I.tb = 0;
    I.seqlen = p.N;
    if (VARLEN) {
        // no cu_seqlens: B sequences of N tokens each ([B, N, H, d] tensors)
        const int a = p.cu_seqlens ? __ldg(p.cu_seqlens + I.b) : I.b * p.N;
        const int e = p.cu_seqlens ? __ldg(p.cu_seqlens + I.b + 1) : a + p.N;
        I.tb = a;
        I.seqlen = max(0, min(e - a, p.N));
    }
    int kvl = I.seqlen;
    I.tbk = I.tb;
    I.coff = 0;
    if (VARLEN && p.cu_seqlens_k) {  // its own key range; causal: the queries are the last len_q positions
        I.tbk = __ldg(p.cu_seqlens_k + I.b);
        kvl = max(0, __ldg(p.cu_seqlens_k + I.b + 1) - I.tbk);
        I.coff = kvl - I.seqlen;
    }
    if constexpr (RECT) kvl = p.Nk;
    if (!VARLEN && p.kv_lens) kvl = min(max(__ldg(p.kv_lens + I.b), 0), key_count(p));
    I.kvl = kvl;
    const int key0 = I.kt * C::BC;
    const int iend = ((VARLEN ? I.seqlen : p.N) + C::BR - 1) / C::BR;
    I.i0 = CAUSAL ? (RECT ? max(0, key0 - causal_offset(p)) : VARLEN ? max(0, key0 - I.coff) : key0) / C::BR : 0;
    if constexpr (SPARSE) {
        // the block's query blocks, without those entirely above the causal
        // diagonal (all query rows before the block's first key)
        constexpr int R = 128 / C::BR;
        const int nnz = __ldg(p.col_ptr + p.nkb);
        int off = min(max(__ldg(p.col_ptr + I.kt), 0), nnz);
        int cnt = min(max(min(__ldg(p.col_ptr + I.kt + 1), nnz) - off, 0), p.nqb);
        if (CAUSAL)
            while (cnt > 0 && (__ldg(p.row_idx + off) + 1) * 128 <= key0) {
                ++off;
                --cnt;
            }
        I.i0 = off;
        I.ni = (key0 >= kvl) ? 0 : cnt * R;
    } else if constexpr (WINDOW) {
        // query rows that see some key of the block: [key0 - right, last key + left]
        int ie = iend;
        if (p.win_right >= 0) I.i0 = max(I.i0, max(0, key0 - p.win_right) / C::BR);
        if (p.win_left >= 0 && key0 < kvl) ie = min(ie, (min(key0 + C::BC, kvl) - 1 + p.win_left) / C::BR + 1);
        I.ni = (key0 >= kvl) ? 0 : max(ie - I.i0, 0);
    } else {
        I.ni = (key0 >= kvl) ? 0 : max(iend - I.i0, 0);
    }
    I.n = I.ni * gper;
    return I;
}
// Query head row bhq and query block i of consecutive steps of an item:
// start with (qh0, i0), advance once per step (one query head: i = i0 + s).
// Block-sparse: query head row and query block (in C::BR units) of step s.
template <class C>
__device__ __forceinline__ void sparse_step(const Item& I, const BwdParamsSparse& p, int s, int& bhq, int& i) {
    constexpr int R = 128 / C::BR;
    const int h = s / I.ni, local = s - h * I.ni;
    bhq = I.qh0 + h;
    i = min(max(__ldg(p.row_idx + I.i0 + local / R), 0), p.nqb - 1) * R + local % R;
}

template <bool GQA>
__device__ __forceinline__ void step_next(const Item& I, int& bhq, int& i) {
    ++i;
    if (GQA && i == I.i0 + I.ni) {
        i = I.i0;
        ++bhq;
    }
}

template <bool OUT_F32>
__device__ __forceinline__ void store_chunk32(void* base, size_t elem_off, const float (&v)[32]) {
    if constexpr (OUT_F32) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + elem_off);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + elem_off);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
    }
}

// ---- MMA groups (the MMA warp elects one lane, which issues the whole group) ----
// All descriptors arrive as precomputed bases; per-MMA offsets are constants.
// S^T = K_j Q_i^T  or  dP^T = V_j dO_i^T  (K-major operands)
template <class C>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint64_t kv_desc, uint64_t q_desc) {
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk)
            mma_f16_ss(d_tmem, desc_add(kv_desc, (kk / 4) * C::K_BOX + (kk % 4) * 32),
                       desc_add(q_desc, (kk / 4) * C::Q_BOX + (kk % 4) * 32), C::IDESC_S, kk > 0);
    }
    __syncwarp();
}
// The same products with K_j or V_j from TMEM (kv_tmem: its first column;
// K-major, two head-dim elements per column, 8 columns per 16-wide K step)
template <class C>
__device__ __forceinline__ void mma_scores_t(uint32_t d_tmem, uint32_t kv_tmem, uint64_t q_desc) {
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk)
            mma_f16_ts(d_tmem, kv_tmem + kk * 8, desc_add(q_desc, (kk / 4) * C::Q_BOX + (kk % 4) * 32), C::IDESC_S,
                       kk > 0 ? 1u : 0u);
    }
    __syncwarp();
}
// TMEM column of the packed P^T for queries [16 kk, 16 kk + 16): each compute
// warpgroup h writes its half at the start of its own S^T columns (never into
// columns the other warpgroup may still be reading).
template <class C>
__device__ __forceinline__ constexpr uint32_t p_col(int kk) {
    return (uint32_t)(((kk * 16) / C::HALF) * C::HALF + ((kk * 16) % C::HALF) / 2);
}
// dV_j (+)= P^T dO_i  (P^T from TMEM, dO_i MN-major: do_mn = MN-major base)
template <class C>
__device__ __forceinline__ void mma_dv(uint32_t tmem, uint32_t s_tmem, uint64_t do_mn, bool acc) {
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < C::BR / 16; ++kk)
            mma_f16_ts(tmem + C::TM_DV, s_tmem + p_col<C>(kk), desc_add(do_mn, kk * 2048), C::IDESC_ACC,
                       (acc || kk > 0) ? 1u : 0u);
    }
    __syncwarp();
}
// dK_j (+)= dS^T Q_i  (dS^T K-major in smem, Q_i MN-major)
template <class C>
__device__ __forceinline__ void mma_dk(uint32_t tmem, uint64_t ds_k, uint64_t q_mn, bool acc) {
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < C::BR / 16; ++kk)
            mma_f16_ss(tmem + C::TM_DK, desc_add(ds_k, (kk / 4) * C::DS_BOX + (kk % 4) * 32),
                       desc_add(q_mn, kk * 2048), C::IDESC_ACC, (acc || kk > 0) ? 1u : 0u);
    }
    __syncwarp();
}
// d=128: dQ^T = K_j^T dS^T ; d=64: dQ = dS K_j  (both operands MN-major)
template <class C>
__device__ __forceinline__ void mma_dq(uint32_t d_tmem, uint64_t k_mn, uint64_t ds_mn) {
    if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < C::BC / 16; ++kk) {
            const uint64_t dk = desc_add(k_mn, kk * 2048);
            const uint64_t ds = desc_add(ds_mn, kk * 2048);
            if (C::D == 128)
                mma_f16_ss(d_tmem, dk, ds, C::IDESC_DQ, kk > 0);
            else
                mma_f16_ss(d_tmem, ds, dk, C::IDESC_DQ, kk > 0);
        }
    }
    __syncwarp();
}

// Copy key row `kr` of the K_j and V_j tiles (128-byte-swizzle boxes of 64
// head-dim elements: 16-byte chunk c of row r at chunk c ^ (r & 7)) into the
// calling warp's TMEM lane, bf16 pairs in head-dim order: the K-major A
// operand layout of tcgen05.mma with A in TMEM.
template <class C>
__device__ __forceinline__ void copy_kv_to_tmem(const uint8_t* smem, uint32_t t_lane, int kr) {
#pragma unroll 1
    for (int t = 0; t < 2; ++t) {
        const uint8_t* tile = smem + (t ? C::OFF_V : C::OFF_K);
#pragma unroll 1
        for (int bx = 0; bx < C::NBOX; ++bx) {
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int off = bx * C::K_BOX + kr * 128 + ((c ^ (kr & 7)) * 16);
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (dcheck(chk::range_ok(off, 16, C::K_TILE), kErrCheckSmem))
                    u = *reinterpret_cast<const uint4*>(tile + off);
                w[4 * c] = u.x;
                w[4 * c + 1] = u.y;
                w[4 * c + 2] = u.z;
                w[4 * c + 3] = u.w;
            }
            tmem_st32(t_lane + (t ? C::TM_V : C::TM_K) + bx * 32, w);
        }
    }
}

template <class C, bool CAUSAL, bool OUT_F32, bool GQA, bool VARLEN = false, bool WINDOW = false,
          bool SPARSE = false, bool RECT = false, bool DET = false>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
               const __grid_constant__ CUtensorMap tdq, const KernelParamsT<WINDOW, SPARSE, RECT, DET> p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto BAR = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
    FA_CHECK_BIND(p.err);

    if (threadIdx.x == 0) {
        mbar_init(BAR(C::B_KVFULL), 1);
        mbar_init(BAR(C::B_KVEMPTY), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(BAR(C::B_QFULL + s), 1);
            mbar_init(BAR(C::B_QEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(C::B_SFULL + s), 1);
            mbar_init(BAR(C::B_DPFULL + s), 1);
            mbar_init(BAR(C::B_PFULL + s), 256);
            mbar_init(BAR(C::B_DSFULL + s), 256);
            mbar_init(BAR(C::B_DSEMPTY + s), 1);
            mbar_init(BAR(C::B_DQFULL + s), 1);
            mbar_init(BAR(C::B_DQEMPTY + s), 128);
        }
        mbar_init(BAR(C::B_ACCFULL), 1);
        mbar_init(BAR(C::B_ACCEMPTY), 256);
        mbar_init(BAR(C::B_DONE), 1);
        mbar_init(BAR(C::B_KVTFULL), 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
        tmem_relinquish();
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            prefetch_tmap(&tdo);
            prefetch_tmap(&tdq);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        int st = 0;
        uint32_t ph = 0, kve = 0;
        bool ok = true;
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item<C, CAUSAL, GQA, VARLEN, WINDOW, SPARSE, RECT, DET>(it, p);
            if (I.n == 0) continue;
            if (!(ok = wait_bounded_warp(BAR(C::B_KVEMPTY), kve ^ 1, abort_flag, p.err, kErrWaitBwdProducer))) break;
            kve ^= 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR(C::B_KVFULL), 2 * C::K_TILE);
                for (int bx = 0; bx < C::NBOX; ++bx) {
                    const int c1 = VARLEN ? I.kvh : I.kt * C::BC, c2 = VARLEN ? I.tbk + I.kt * C::BC : I.bh;
                    tma_load_3d(sbase + C::OFF_K + bx * C::K_BOX, &tk, BAR(C::B_KVFULL), bx * 64, c1, c2);
                    tma_load_3d(sbase + C::OFF_V + bx * C::K_BOX, &tv, BAR(C::B_KVFULL), bx * 64, c1, c2);
                }
            }
            __syncwarp();
            int bhq = I.qh0, i = I.i0;
            for (int s = 0; s < I.n; ++s, step_next<GQA>(I, bhq, i)) {
                if constexpr (SPARSE) sparse_step<C>(I, p, s, bhq, i);
                if (!(ok = wait_bounded_warp(BAR(C::B_QEMPTY + st), ph ^ 1, abort_flag, p.err, kErrWaitBwdProducer))) break;
                if (lane == 0) {
                    const uint32_t bar = BAR(C::B_QFULL + st);
                    mbar_arrive_expect_tx(bar, 2 * C::Q_TILE + C::STAT_BYTES);
                    for (int bx = 0; bx < C::NBOX; ++bx) {
                        const int c1 = VARLEN ? bhq : i * C::BR, c2 = VARLEN ? I.tb + i * C::BR : bhq;
                        tma_load_3d(sbase + C::OFF_Q + st * C::Q_TILE + bx * C::Q_BOX, &tq, bar, bx * 64, c1, c2);
                        tma_load_3d(sbase + C::OFF_DO + st * C::Q_TILE + bx * C::Q_BOX, &tdo, bar, bx * 64, c1, c2);
                    }
                    const size_t roff = (size_t)(VARLEN ? bhq * p.B + I.b : bhq) * p.Np + (size_t)i * C::BR;
                    bulk_load(sbase + C::OFF_STAT + st * C::STAT_BYTES, p.lse2 + roff, C::BR * 4, bar);
                    bulk_load(sbase + C::OFF_STAT + st * C::STAT_BYTES + C::BR * 4, p.dvec + roff, C::BR * 4, bar);
                }
                __syncwarp();
                if (++st == C::STAGES) { st = 0; ph ^= 1; }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Per item (one TMEM slot):
        //   prologue: S(0), dP(0)
        //   step s:   dV(s) | S(s+1) | dQ(s), dK(s) | dP(s+1) once dQ(s) is drained
        // so the compute warpgroups have the next step's S in flight while they
        // form dS(s), and dQ(s), which the next dP waits for, goes first.
        int st = 0, st_ahead = 0;  // Q ring stage of step s / of the next step to open
        uint32_t qph = 0, qph_ahead = 0, kvph = 0, aeph = 0;
        uint32_t pph[2] = {0, 0}, dsph[2] = {0, 0}, dqeph[2] = {0, 0};
        const uint64_t k_kd = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
        const uint64_t v_kd = sdesc_sw128(sbase + C::OFF_V, 16, 1024);
        const uint64_t k_mn = sdesc_sw128(sbase + C::OFF_K, C::K_BOX, 1024);
        const uint64_t q_kd0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
        const uint64_t q_mn0 = sdesc_sw128(sbase + C::OFF_Q, C::Q_BOX, 1024);
        const uint64_t do_kd0 = sdesc_sw128(sbase + C::OFF_DO, 16, 1024);
        const uint64_t do_mn0 = sdesc_sw128(sbase + C::OFF_DO, C::Q_BOX, 1024);
        const uint64_t ds_kd0 = sdesc_sw128(sbase + C::OFF_DS, 16, 1024);
        const uint64_t ds_mn0 = sdesc_sw128(sbase + C::OFF_DS, C::DS_BOX, 1024);
        bool ok = true;
        // open_step(slot): wait for the next step's Q/dO stage and issue its S
        auto open_step = [&](int slot) -> bool {
            if (!wait_bounded_warp(BAR(C::B_QFULL + st_ahead), qph_ahead, abort_flag, p.err, kErrWaitBwdMma)) return false;
            tc_fence_after();
            if constexpr (C::KV_TMEM)
                mma_scores_t<C>(tmem + C::s_col(slot), tmem + C::TM_K, desc_add(q_kd0, st_ahead * C::Q_TILE));
            else
                mma_scores<C>(tmem + C::s_col(slot), k_kd, desc_add(q_kd0, st_ahead * C::Q_TILE));
            mma_commit_w(BAR(C::B_SFULL + slot));
            if (++st_ahead == C::STAGES) { st_ahead = 0; qph_ahead ^= 1; }
            return true;
        };
        // issue_dp(slot, stage): dP^T of the step held in `stage` into the slot's X
        // columns, once the dQ previously held there has been drained
        auto issue_dp = [&](int slot, int stage) -> bool {
            if (C::DQ_ALIAS) {
                if (!wait_bounded_warp(BAR(C::B_DQEMPTY + slot), dqeph[slot] ^ 1, abort_flag, p.err, kErrWaitBwdMma))
                    return false;
                dqeph[slot] ^= 1;
            }
            tc_fence_after();
            if constexpr (C::KV_TMEM)
                mma_scores_t<C>(tmem + C::x_col(slot), tmem + C::TM_V, desc_add(do_kd0, stage * C::Q_TILE));
            else
                mma_scores<C>(tmem + C::x_col(slot), v_kd, desc_add(do_kd0, stage * C::Q_TILE));
            mma_commit_w(BAR(C::B_DPFULL + slot));
            return true;
        };
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item<C, CAUSAL, GQA, VARLEN, WINDOW, SPARSE, RECT, DET>(it, p);
            if (I.n == 0) continue;
            if (!(ok = wait_bounded_warp(BAR(C::B_KVFULL), kvph, abort_flag, p.err, kErrWaitBwdMma))) break;
            if constexpr (C::KV_TMEM)  // the drain warps have copied K_j, V_j into TMEM
                if (!(ok = wait_bounded_warp(BAR(C::B_KVTFULL), kvph, abort_flag, p.err, kErrWaitBwdMma))) break;
            kvph ^= 1;
            // prologue: S of the first NSLOT steps, then their dP
            for (int s = 0; s < C::NSLOT && s < I.n && ok; ++s) ok = open_step(s);
            for (int s = 0; s < C::NSLOT && s < I.n && ok; ++s) ok = issue_dp(s, (st + s) % C::STAGES);
            if (!ok) break;
            for (int s = 0; s < I.n; ++s) {
                const int slot = s % C::NSLOT;
                const int dsb = s & 1;
                // dV(s)
                if (!(ok = wait_bounded_warp(BAR(C::B_PFULL + slot), pph[slot], abort_flag, p.err, kErrWaitBwdMma))) break;
                pph[slot] ^= 1;
                if (s == 0) {
                    if (!(ok = wait_bounded_warp(BAR(C::B_ACCEMPTY), aeph ^ 1, abort_flag, p.err, kErrWaitBwdMma))) break;
                    aeph ^= 1;
                }
                tc_fence_after();
                mma_dv<C>(tmem, tmem + C::s_col(slot), desc_add(do_mn0, st * C::Q_TILE), s > 0);
                // S(s + NSLOT) into this slot (its P(s) is consumed by dV(s), issued before)
                if (s + C::NSLOT < I.n && !(ok = open_step(slot))) break;
                // dK(s), dQ(s)
                if (!(ok = wait_bounded_warp(BAR(C::B_DSFULL + slot), dsph[slot], abort_flag, p.err, kErrWaitBwdMma))) break;
                dsph[slot] ^= 1;
                const int dqs = C::DQ_ALIAS ? slot : 0;
                if (!C::DQ_ALIAS) {  // separate dQ region: previous tile drained?
                    if (!(ok = wait_bounded_warp(BAR(C::B_DQEMPTY), dqeph[0] ^ 1, abort_flag, p.err, kErrWaitBwdMma))) break;
                    dqeph[0] ^= 1;
                }
                tc_fence_after();
                mma_dq<C>(tmem + C::dq_col(slot), k_mn, desc_add(ds_mn0, dsb * C::DS_TILE));
                mma_commit_w(BAR(C::B_DQFULL + dqs));
                mma_dk<C>(tmem, desc_add(ds_kd0, dsb * C::DS_TILE), desc_add(q_mn0, st * C::Q_TILE), s > 0);
                mma_commit_w(BAR(C::B_QEMPTY + st));
                mma_commit_w(BAR(C::B_DSEMPTY + dsb));
                // dP(s+1) for steps past the prologue
                if (s + 1 < I.n && s + 1 >= C::NSLOT && !(ok = issue_dp((s + 1) % C::NSLOT, (st + 1) % C::STAGES)))
                    break;
                if (++st == C::STAGES) { st = 0; qph ^= 1; }
            }
            if (!ok) break;
            mma_commit_w(BAR(C::B_KVEMPTY));
            mma_commit_w(BAR(C::B_ACCFULL));
        }
        (void)qph;
        mma_commit_w(BAR(C::B_DONE));
        wait_bounded_warp(BAR(C::B_DONE), 0, abort_flag, p.err, kErrWaitDrain);
    } else if (warp < 8) {
        // ------------------------------------------------------------ compute warpgroups
        const int h = warp >> 2;  // query-column half
        const int wq = warp & 3;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int kr = wq * 32 + lane;  // key row of this thread within the block
        int st = 0;
        uint32_t qph = 0, acph = 0;
        uint32_t sph[2] = {0, 0}, dpph[2] = {0, 0}, dseph[2] = {0, 0};
        bool ok = true;
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item<C, CAUSAL, GQA, VARLEN, WINDOW, SPARSE, RECT, DET>(it, p);
            const int key = I.kt * C::BC + kr;
            // dK, dV row: [B,Hkv,N,d], or token-major [total, Hkv, d] for packed sequences
            const int nkeys = key_count(p);
            const size_t krow = VARLEN ? (size_t)(I.tbk + key) * p.Hkv + I.kvh : (size_t)I.bh * nkeys + key;
            if (I.n == 0) {  // no query sees the key block: zero gradients for its keys
                // (beyond kv_len; packed: a sequence with keys but no queries)
                if (VARLEN ? key < I.kvl : key < nkeys) {
                    float z[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] = 0.f;
                    if (GQA && p.gsplit > 1) {
                        float* part = p.dkv_part + (size_t)(I.sub * 2 + h) * p.B * p.Hkv * nkeys * C::D;
#pragma unroll
                        for (int c = 0; c < C::D; c += 32) store_chunk32<true>(part, krow * C::D + c, z);
                    } else {
                        void* dst = h ? p.dk : p.dv;
#pragma unroll
                        for (int c = 0; c < C::D; c += 32) store_chunk32<OUT_F32>(dst, krow * C::D + c, z);
                    }
                }
                continue;
            }
            int bhq = I.qh0, i = I.i0;
            for (int s = 0; s < I.n; ++s, step_next<GQA>(I, bhq, i)) {
                if constexpr (SPARSE) sparse_step<C>(I, p, s, bhq, i);
                const int slot = s % C::NSLOT;
                const int dsb = s & 1;
                const int q0 = i * C::BR + h * C::HALF;  // first query column of this half
                // statistics of this stage (LSE*log2e, D) -- readable once the stage is full
                if (!(ok = wait_bounded_warp(BAR(C::B_QFULL + st), qph, abort_flag, p.err, kErrWaitBwdCompute))) break;
                const float* lse2 = reinterpret_cast<const float*>(smem + C::OFF_STAT + st * C::STAT_BYTES) + h * C::HALF;
                const float* dvec = lse2 + C::BR;
                if (!(ok = wait_bounded_warp(BAR(C::B_SFULL + slot), sph[slot], abort_flag, p.err, kErrWaitBwdCompute))) break;
                sph[slot] ^= 1;
                tc_fence_after();
                uint32_t sr[C::HALF];
                if constexpr (C::HALF == 32)
                    tmem_ld32_wait(tmem + lane_off + C::s_col(slot) + h * C::HALF, *reinterpret_cast<uint32_t(*)[32]>(sr));
                else
                    tmem_ld64_wait(tmem + lane_off + C::s_col(slot) + h * C::HALF, *reinterpret_cast<uint32_t(*)[64]>(sr));
                const int coff = VARLEN ? I.coff : causal_offset(p);  // 0 unless rectangular / packed q != k
                bool need_mask = (I.kt * C::BC + C::BC > I.kvl) || (CAUSAL && I.kt * C::BC + C::BC - 1 > i * C::BR + coff);
                if constexpr (WINDOW)  // some pair of the tile outside the window
                    need_mask = need_mask || (p.win_right >= 0 && I.kt * C::BC + C::BC - 1 > i * C::BR + p.win_right) ||
                                (p.win_left >= 0 && I.kt * C::BC < i * C::BR + C::BR - 1 - p.win_left);
                const bool key_ok = key < I.kvl;
                float pv[C::HALF];
                const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
                for (int c = 0; c < C::HALF; c += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
                    const float2 x0 = ffma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2,
                                            make_float2(-l4.x, -l4.y));
                    const float2 x1 = ffma2(make_float2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), sl2,
                                            make_float2(-l4.z, -l4.w));
                    pv[c + 0] = ex2_approx(x0.x);
                    pv[c + 1] = ex2_approx(x0.y);
                    pv[c + 2] = ex2_approx(x1.x);
                    pv[c + 3] = ex2_approx(x1.y);
                }
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < C::HALF; ++c) {
                        const int q = q0 + c;
                        bool off = !key_ok || (CAUSAL && key > q + coff);
                        if constexpr (WINDOW)
                            off = off || (p.win_right >= 0 && key > q + p.win_right) || (p.win_left >= 0 && key < q - p.win_left);
                        if (off) pv[c] = 0.f;
                    }
                }
                // P^T (bf16) over this half's S^T columns, as the A operand of dV += P^T dO
                {
                    uint32_t w[C::HALF / 2];
#pragma unroll
                    for (int c = 0; c < C::HALF / 2; ++c) w[c] = pack_bf16x2(pv[2 * c], pv[2 * c + 1]);
                    const uint32_t tp = tmem + lane_off + C::s_col(slot) + h * C::HALF;
                    if constexpr (C::HALF == 32) {
                        tmem_st16(tp, *reinterpret_cast<uint32_t(*)[16]>(w));
                    } else {
                        tmem_st32(tp, *reinterpret_cast<uint32_t(*)[32]>(w));
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(BAR(C::B_PFULL + slot));
                // dS = P (dP - D)
                if (!(ok = wait_bounded_warp(BAR(C::B_DPFULL + slot), dpph[slot], abort_flag, p.err, kErrWaitBwdCompute))) break;
                dpph[slot] ^= 1;
                tc_fence_after();
                if (!(ok = wait_bounded_warp(BAR(C::B_DSEMPTY + dsb), dseph[dsb] ^ 1, abort_flag, p.err, kErrWaitBwdCompute))) break;
                dseph[dsb] ^= 1;
                // write dS^T row `kr` (queries h*HALF .. +HALF) into the swizzled tile,
                // 32 dP columns at a time
#pragma unroll
                for (int cc = 0; cc < C::HALF; cc += 32) {
                    uint32_t dr[32];
                    tmem_ld32_wait(tmem + lane_off + C::x_col(slot) + h * C::HALF + cc, dr);
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        const int c = cc + c8;
                        const int qc = h * C::HALF + c;  // query column within the block
                        const int box = qc / 64, chunk = (qc % 64) / 8;
                        const float4 d0 = *reinterpret_cast<const float4*>(dvec + c);
                        const float4 d1 = *reinterpret_cast<const float4*>(dvec + c + 4);
                        const float g0 = pv[c + 0] * (__uint_as_float(dr[c8 + 0]) - d0.x);
                        const float g1 = pv[c + 1] * (__uint_as_float(dr[c8 + 1]) - d0.y);
                        const float g2 = pv[c + 2] * (__uint_as_float(dr[c8 + 2]) - d0.z);
                        const float g3 = pv[c + 3] * (__uint_as_float(dr[c8 + 3]) - d0.w);
                        const float g4 = pv[c + 4] * (__uint_as_float(dr[c8 + 4]) - d1.x);
                        const float g5 = pv[c + 5] * (__uint_as_float(dr[c8 + 5]) - d1.y);
                        const float g6 = pv[c + 6] * (__uint_as_float(dr[c8 + 6]) - d1.z);
                        const float g7 = pv[c + 7] * (__uint_as_float(dr[c8 + 7]) - d1.w);
                        const uint4 v = make_uint4(pack_bf16x2(g0, g1), pack_bf16x2(g2, g3), pack_bf16x2(g4, g5),
                                                   pack_bf16x2(g6, g7));
                        const int dso = dsb * C::DS_TILE + box * C::DS_BOX + kr * 128 + ((chunk ^ (kr & 7)) * 16);
                        if (dcheck(chk::range_ok(dso, 16, 2 * C::DS_TILE), kErrCheckSmem))
                            *reinterpret_cast<uint4*>(smem + C::OFF_DS + dso) = v;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(BAR(C::B_DSFULL + slot));
                if (++st == C::STAGES) { st = 0; qph ^= 1; }
            }
            if (!ok) break;
            // epilogue: warpgroup 0 writes dV_j, warpgroup 1 writes scale * dK_j
            if (!(ok = wait_bounded_warp(BAR(C::B_ACCFULL), acph, abort_flag, p.err, kErrWaitBwdCompute))) break;
            acph ^= 1;
            tc_fence_after();
            const float mul = h ? p.scale : 1.f;
            void* dst = h ? p.dk : p.dv;
            const bool to_part = GQA && !VARLEN && p.gsplit > 1;  // split group: float32 partial slice
            float* part = to_part ? p.dkv_part + (size_t)(I.sub * 2 + h) * p.B * p.Hkv * nkeys * C::D : nullptr;
            const uint32_t tacc = tmem + lane_off + (h ? C::TM_DK : C::TM_DV);
#pragma unroll 1
            for (int c = 0; c < C::D; c += 32) {
                uint32_t a[32];
                tmem_ld32_wait(tacc + c, a);
                float f[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(a[e]) * mul;
                if (key < (VARLEN ? I.kvl : nkeys)) {
                    if (to_part)
                        store_chunk32<true>(part, krow * C::D + c, f);
                    else
                        store_chunk32<OUT_F32>(dst, krow * C::D + c, f);
                }
            }
            tc_fence_before();
            mbar_arrive(BAR(C::B_ACCEMPTY));
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ dQ drain warps
        const int wq = warp - kDqWarp0;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t stage = sbase + C::OFF_DQ + wq * C::DQ_WARP_BYTES;
        float* stage_f = reinterpret_cast<float*>(smem + C::OFF_DQ + wq * C::DQ_WARP_BYTES);
        uint32_t dqph[2] = {0, 0}, kvph = 0;
        bool ok = true;
        // DET: pend[j] is the turn counter of the write issued j + 1 steps ago;
        // it is passed on once that write has completed (kDetLag steps later,
        // or at the item's end)
        int* pend[kDetLag];
#pragma unroll
        for (int j = 0; j < kDetLag; ++j) pend[j] = nullptr;
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item<C, CAUSAL, GQA, VARLEN, WINDOW, SPARSE, RECT, DET>(it, p);
            if (C::KV_TMEM && I.n > 0) {
                // K_j, V_j rows of this warp's lanes into TMEM.  The previous item's
                // S and dP products, the only readers, were issued before its last dQ
                // product, whose completion this warp has already waited for.
                if (!(ok = wait_bounded_warp(BAR(C::B_KVFULL), kvph, abort_flag, p.err, kErrWaitBwdDq))) break;
                kvph ^= 1;
                copy_kv_to_tmem<C>(smem, tmem + lane_off, wq * 32 + lane);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(BAR(C::B_KVTFULL));
            }
            int bhq = I.qh0, i = I.i0;
            for (int s = 0; s < I.n; ++s, step_next<GQA>(I, bhq, i)) {
                if constexpr (SPARSE) sparse_step<C>(I, p, s, bhq, i);
                const int dqs = C::DQ_ALIAS ? (s % C::NSLOT) : 0;
                if (!(ok = wait_bounded_warp(BAR(C::B_DQFULL + dqs), dqph[dqs], abort_flag, p.err, kErrWaitBwdDq))) break;
                dqph[dqs] ^= 1;
                tc_fence_after();
                uint32_t v[64];
                tmem_ld64_wait(tmem + lane_off + C::dq_col(dqs), v);
                tc_fence_before();
                mbar_arrive(BAR(C::B_DQEMPTY + dqs));
                // the previous reduction of this warp must have finished reading the staging
                if (lane == 0) {
                    bulk_wait_group_read<0>();
                    if constexpr (DET) {
                        if (pend[kDetLag - 1]) {
                            bulk_wait_group<kDetLag - 1>();  // all but the last kDetLag - 1 writes are done
                            fence_proxy_async_global();
                            red_release_gpu_add(pend[kDetLag - 1], 1);
                        }
                    }
                }
                if constexpr (DET) {
#pragma unroll
                    for (int j = kDetLag - 1; j > 0; --j) pend[j] = pend[j - 1];
                    pend[0] = nullptr;
                }
                __syncwarp();
                if constexpr (C::D == 128) {
                    // lane = head-dim index (wq*32 + lane); column = query. Stage [64 q][32 d].
                    if (dcheck(chk::range_ok(63 * 32 * 4 + lane * 4, 4, C::DQ_WARP_BYTES), kErrCheckSmem))
#pragma unroll
                        for (int q = 0; q < 64; ++q) stage_f[q * 32 + lane] = __uint_as_float(v[q]);
                } else {
                    // lane = query (wq*32 + lane); column = head dim.  Two [32 q][32 d]
                    // boxes in the 128-byte-swizzle layout: 16-byte chunk c of row r
                    // sits at chunk c ^ (r & 7), so eight consecutive lanes cover all
                    // banks, and every register index stays a compile-time constant;
                    // the tensor reduction undoes the swizzle on its way to global memory
                    uint8_t* stage_b = reinterpret_cast<uint8_t*>(stage_f);
                    if (dcheck(chk::range_ok(4096 + lane * 128 + 7 * 16, 16, C::DQ_WARP_BYTES), kErrCheckSmem))
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<float4*>(stage_b + b * 4096 + lane * 128 + ((c ^ (lane & 7)) * 16)) =
                                make_float4(__uint_as_float(v[32 * b + 4 * c]), __uint_as_float(v[32 * b + 4 * c + 1]),
                                            __uint_as_float(v[32 * b + 4 * c + 2]), __uint_as_float(v[32 * b + 4 * c + 3]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                int row = (VARLEN ? bhq * p.B + I.b : bhq) * p.Np + i * C::BR;
                bool first = false;
                if constexpr (DET) {
                    // the visitors of query block i, in increasing key block order, take
                    // accumulators 0, 1, ..., nacc - 1, 0, ...: a key block writes after
                    // the visitors nacc, 2 nacc, ... places before it; the first stores.
                    // Without block lists they are the key blocks lo .. (i0 and the
                    // window's end grow with the key block)
                    // pos: this key block's place among the query block's visitors
                    int pos;
                    if constexpr (SPARSE) {
                        // block lists: the visitors are the query block's list (ascending;
                        // the causal and key-length cuts only drop its tail); binary search
                        const int qb = (i * C::BR) / 128;
                        int lo = 0;
                        if (lane == 0) {
                            const int nnz = __ldg(p.row_ptr + p.nqb);
                            const int b0 = min(max(__ldg(p.row_ptr + qb), 0), nnz);
                            int hi = min(max(__ldg(p.row_ptr + qb + 1), b0), nnz);
                            lo = b0;
                            while (lo < hi) {  // first position whose key block is >= kt
                                const int mid = (lo + hi) >> 1;
                                if (__ldg(p.col_idx + mid) < I.kt) lo = mid + 1;
                                else hi = mid;
                            }
                            lo -= b0;
                        }
                        pos = __shfl_sync(0xffffffffu, lo, 0);
                    } else {
                        int lo = 0;
                        if constexpr (WINDOW)  // first key block whose window reaches query block i
                            if (p.win_left >= 0) lo = max(0, i * C::BR - p.win_left) / C::BC;
                        pos = I.kt - lo;
                    }
                    const int a = pos % p.nacc;
                    const int srow = VARLEN ? bhq * p.B + I.b : bhq;  // statistics row group of the tile
                    int* turn = p.dq_turn + (((size_t)a * (p.B * p.H) + srow) * p.nqt + i) * 4 + wq;
                    if (!(ok = wait_turn_warp(turn, pos / p.nacc, abort_flag, p.err, kErrWaitBwdDqTurn))) break;
                    pend[0] = turn;
                    row += a * (p.B * p.H * p.Np);
                    first = pos < p.nacc;
                }
                if (lane == 0) {
                    if constexpr (DET) fence_proxy_async_global();
                    if constexpr (C::D == 128) {
                        if (first) tma_store_2d(&tdq, stage, wq * 32, row);
                        else tma_reduce_add_2d(&tdq, stage, wq * 32, row);
                    } else {
                        if (first) {
                            tma_store_2d(&tdq, stage, 0, row + wq * 32);
                            tma_store_2d(&tdq, stage + 4096, 32, row + wq * 32);
                        } else {
                            tma_reduce_add_2d(&tdq, stage, 0, row + wq * 32);
                            tma_reduce_add_2d(&tdq, stage + 4096, 32, row + wq * 32);
                        }
                    }
                    bulk_commit_group();
                }
                __syncwarp();
            }
            if constexpr (DET) {
                // pass the item's last turns on before the next item's waits
                if (lane == 0) {
                    bulk_wait_group<0>();
                    fence_proxy_async_global();
#pragma unroll
                    for (int j = kDetLag - 1; j >= 0; --j)
                        if (pend[j]) red_release_gpu_add(pend[j], 1);
                }
#pragma unroll
                for (int j = 0; j < kDetLag; ++j) pend[j] = nullptr;
                __syncwarp();
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kProducerWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <class C, bool CAUSAL, bool OUT_F32, bool GQA = false, bool VARLEN = false, bool WINDOW = false,
          bool SPARSE = false, bool RECT = false, bool DET = false>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& tdo, const CUtensorMap& tdq, const KernelParamsT<WINDOW, SPARSE, RECT, DET>& p,
                   int grid, cudaStream_t stream) {
    auto kern = bwd_kernel<C, CAUSAL, OUT_F32, GQA, VARLEN, WINDOW, SPARSE, RECT, DET>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, p);
    return cudaGetLastError();
}

}  // namespace bwd
}  // namespace fa

// Persistent forward kernel of exact tiled attention for sm_103a.
//
// What it computes is Algorithm 1 of the FA-v2 analysis page
// ("解析 FlashAttention（4）：FlashAttention-v2", §4): for a block of query rows
// it walks the key/value blocks keeping, per row, the running maximum m, the
// running sum l and the unnormalised output O; it rescales the old state by
// exp(m_old - m_new) (multiplication, as in that page's §2.3 scalar derivation
// and the running-state formulas of the attention-kernels wiki §01), and
// finally writes O / l and LSE = m + log l (§4 steps 6-7).  Masks follow
// chapter 18 §18.2.2 (causal M_ij = -inf for j > i; padding masks columns,
// Table 18-3); fully masked key blocks are skipped (§18.5.2), and a row with
// no visible key gets O = 0, LSE = -inf (wiki §04).
//
// How it maps onto a GB300 SM (one CTA per SM, persistent over work items):
//   * a work item is one (batch, head, pair of 128-row query tiles);
//   * warp 8 (one lane) issues TMA loads of Q (once per item) and a ring of
//     K and V tiles (128-byte swizzle, one box per 128 bytes of head dim);
//   * warp 9 (one lane) issues tcgen05.mma: S_t = Q_t K_j^T into TMEM, then
//     O_t += P_t V_j with P_t read from TMEM, alternating the two query tiles
//     so the tensor core works on one tile while the other is in softmax;
//   * warps 0-3 / 4-7 are the softmax warpgroups of tile 0 / tile 1: one
//     thread per query row (= TMEM lane).  Each loads its S row, applies the
//     mask on boundary blocks, updates (m, l) in the log2 domain, rescales its
//     O row in TMEM only when the max grew by more than kRescaleSlack
//     (conditional rescaling: exact, since O/l and m + log l do not depend on
//     which reference max was used), writes P = 2^(S*c - m) back over its S
//     columns as packed bf16 (or E4M3) for the P V MMA, and at the end of the
//     item normalises O and stores O and LSE.
//   TMEM (512 columns): S0 | S1 | O0 | O1 (fp32), P_t aliased on S_t.
//   FP8 variant: Q8 K8 with per-64-row block scales s_q, s_k folded into the
//   softmax multiplier, V's per-block scale folded into the E4M3 P operand.
#pragma once
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace fa {
namespace fwd {

constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Conditional rescaling slack in the log2 domain: P values may reach 2^8
// before the reference max is moved (bf16 path).  The FP8 path keeps the exact
// max so that P <= 1 fits the E4M3 range after the value-scale fold.
constexpr float kRescaleSlack = 8.0f;
// FP8: the probabilities enter P V as E4M3 codes of P * w, w = (value-block
// scale / head's largest value-block scale) * kFp8Fold.  The fold leaves room
// for P up to 2^kFp8Slack (4 * 112 = 448, the E4M3 maximum), so the exact
// reference max taken first needs to move (and O be rescaled) only when a
// row's max grows by more than kFp8Slack.
constexpr float kFp8Slack = 2.0f;
constexpr float kFp8Fold = 112.0f;
// bf16 path: the block's row max is taken first and the reference max moves
// (with O rescaled) only when it grew by more than kRescaleSlack; P is then
// written to TMEM in two halves of the block, and the MMA warp issues the P V
// product of the first half while the softmax computes the second.

template <int D_, int BC_, bool FP8_, bool SPLIT_ = false>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int BC = BC_;
    static constexpr bool FP8 = FP8_;
    // SPLIT: float32 inputs carried as bf16 hi + lo parts; S = Qh Kh^T + Qh Kl^T + Ql Kh^T
    static constexpr bool SPLIT = SPLIT_;
    static constexpr int NPART = SPLIT ? 2 : 1;
    static constexpr int BR = 128;   // query rows per tile (= TMEM lanes)
    static constexpr int QT = 2;     // query tiles per CTA work item
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROW_BYTES = D * ELEM;
    static constexpr int NBOX = ROW_BYTES / 128;  // 128-byte swizzle boxes along d
    static constexpr int BOX_ELEMS = 128 / ELEM;
    static constexpr int Q_BOX = BR * 128;
    static constexpr int KV_BOX = BC * 128;
    static constexpr int Q_TILE = BR * ROW_BYTES;
    static constexpr int KV_TILE = BC * ROW_BYTES;
    // K is needed a step earlier than V (S(j+1) is issued before PV(j+1)), so it
    // gets the deeper ring when shared memory allows
    static constexpr int KV_BUDGET = 232448 - 2048 - NPART * QT * Q_TILE;
    static constexpr int VSTAGES = (KV_TILE >= 32768 || SPLIT) ? 2 : 3;
    static constexpr int KSTAGES_FIT = (KV_BUDGET - VSTAGES * KV_TILE) / (NPART * KV_TILE);
    static constexpr int KSTAGES = KSTAGES_FIT > 4 ? 4 : KSTAGES_FIT;
    static_assert(KSTAGES >= 2, "K ring");
    static constexpr int KSTEP = 32 / ELEM;         // K elements per MMA instruction
    static constexpr int S_STEPS = ROW_BYTES / 32;  // MMAs per S tile
    static constexpr int PV_STEPS = BC / KSTEP;     // MMAs per P V
    static constexpr int TM_S0 = 0, TM_S1 = BC, TM_O0 = 2 * BC, TM_O1 = 2 * BC + D;
    static constexpr int TM_COLS = 512;
    static_assert(2 * BC + 2 * D <= TM_COLS, "TMEM budget");
    // shared memory map (tile bases 1024-byte aligned)
    // Q: [part][tile]; K stage: [part] tiles; V stage: one tile
    static constexpr int OFF_Q = 0;
    static constexpr int K_STAGE = NPART * KV_TILE;
    static constexpr int OFF_K = OFF_Q + NPART * QT * Q_TILE;
    static constexpr int OFF_V = OFF_K + KSTAGES * K_STAGE;
    static constexpr int OFF_BAR = OFF_V + VSTAGES * KV_TILE;
    // barrier indices
    static constexpr int B_QFULL = 0, B_QEMPTY = 2;  // one per query tile
    static constexpr int B_KFULL = 4, B_KEMPTY = 4 + KSTAGES;
    static constexpr int B_VFULL = 4 + 2 * KSTAGES, B_VEMPTY = B_VFULL + VSTAGES;
    static constexpr int B_SFULL = B_VEMPTY + VSTAGES, B_PFULL = B_SFULL + 2;
    static constexpr int B_OFULL = B_PFULL + 2, B_OEMPTY = B_OFULL + 2;
    static constexpr int B_DONE = B_OEMPTY + 2;
    // bf16: P is handed to the MMA warp in two halves of the key block (keys
    // [0, BC/2) complete on B_PHALF, the whole block on B_PFULL), so that the
    // first half of P V runs while the softmax computes the second half
    static constexpr bool SPLITP = !FP8;
    static constexpr int B_PHALF = B_DONE + 1;
    static constexpr int NBAR = B_PHALF + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + base alignment slack
    static constexpr uint32_t FMT = FP8 ? kFmtE4M3 : kFmtBF16;
    // registers per thread of the softmax warpgroups / the issuing warpgroup
    // (setmaxnreg); 2 * 128 * REGS_SOFTMAX + 128 * REGS_ISSUE <= 384 * 168
    static constexpr int REGS_SOFTMAX = FP8 ? 208 : 192, REGS_ISSUE = FP8 ? 88 : 120;
    static constexpr uint32_t IDESC_S = idesc_make(FMT, FMT, 0, 0, 128, BC);
    static constexpr uint32_t IDESC_PV = idesc_make(FMT, FMT, 0, 1, 128, D);
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Item {
    int bh, b, row0, kvl;
    int kvh;    // key/value head row of K, V (b * Hkv + h / group)
    int n[2];   // key blocks of tile 0 / tile 1 in this unit
    int nmax;
    int j0;     // first key block of this unit
    int part;   // partial index of a split unit, -1 for a whole item
};

// Packed variable-length sequences add the head within the sequence and the
// sequence's first token and length.  (A separate type keeps the item of the
// [B, H, N, d] instances at its size: the item lives in local memory there,
// and three more fields cost several percent.)
struct ItemPacked : Item {
    int h, tb, seqlen;
    int tbk, coff;  // first key token; causal offset (keys - queries) of the sequence
};

// Sliding window: each query tile has its own first key block, a[t] blocks
// after the unit's first block j0 (the K / V stream covers the union of the
// two tiles' ranges, which has no gaps).
struct ItemWin : Item {
    int a[2];
};
// Packed sequences under a sliding window.
struct ItemPackedWin : ItemPacked {
    int a[2];
};

// Block-sparse: tile t computes the key blocks col_idx[off[t] .. off[t] +
// n[t] - 1]; the K / V stream is the ascending union of the two lists (nmax
// blocks), walked by BlockMerge in every role.
struct ItemSparse : Item {
    int off[2];
};

template <bool VARLEN, bool WINDOW = false, bool SPARSE = false>
using ItemT = typename std::conditional<
    VARLEN, typename std::conditional<WINDOW, ItemPackedWin, ItemPacked>::type,
    typename std::conditional<WINDOW, ItemWin, typename std::conditional<SPARSE, ItemSparse, Item>::type>::type>::type;

template <bool WINDOW, bool SPARSE = false, bool RECT = false>
using ParamsT = typename std::conditional<
    WINDOW, FwdParamsWin,
    typename std::conditional<SPARSE, FwdParamsSparse,
                              typename std::conditional<RECT, FwdParamsRect, FwdParams>::type>::type>::type;

// Walks the ascending union of the two tiles' key-block lists: each call
// returns the next block and which tiles compute it (a list that is not
// ascending still yields every entry exactly once).
struct BlockMerge {
    const int* l0;
    const int* l1;
    int n0, n1, c0, c1;
    __device__ __forceinline__ int next(bool& a0, bool& a1) {
        const int x0 = c0 < n0 ? __ldg(l0 + c0) : 0x7fffffff;
        const int x1 = c1 < n1 ? __ldg(l1 + c1) : 0x7fffffff;
        const int b = min(x0, x1);
        a0 = c0 < n0 && x0 == b;
        a1 = c1 < n1 && x1 == b;
        c0 += a0;
        c1 += a1;
        return b;
    }
};

__device__ __forceinline__ BlockMerge block_merge(const ItemSparse& I, const FwdParamsSparse& p) {
    BlockMerge m;
    m.l0 = p.col_idx + I.off[0];
    m.l1 = p.col_idx + I.off[1];
    m.n0 = I.n[0];
    m.n1 = I.n[1];
    m.c0 = m.c1 = 0;
    return m;
}

template <class IT>
__host__ __device__ constexpr bool is_packed() { return std::is_base_of<ItemPacked, IT>::value; }
template <class IT>
__host__ __device__ constexpr bool is_window() {
    return std::is_same<IT, ItemWin>::value || std::is_same<IT, ItemPackedWin>::value;
}
template <class IT>
__host__ __device__ constexpr bool is_sparse() { return std::is_same<IT, ItemSparse>::value; }

// First key block of tile t, relative to the unit's j0 (0 without a window).
template <class IT>
__device__ __forceinline__ int item_a(const IT& I, int t) {
    if constexpr (is_window<IT>()) return t ? I.a[1] : I.a[0];
    else return 0;
}

// Key blocks of tile t.  The packed instance reads the field with constant
// indices (its larger item otherwise went to local memory); the others index
// directly, which schedules better.
template <class IT>
__device__ __forceinline__ int item_n(const IT& I, int t) {
    if constexpr (is_packed<IT>() || is_window<IT>() || is_sparse<IT>()) return t ? I.n[1] : I.n[0];
    else return I.n[t];
}

// Query rows of the item's sequence.
template <class IT>
__device__ __forceinline__ int item_rows(const IT& I, const FwdParams& p) {
    if constexpr (is_packed<IT>()) return I.seqlen;
    else return p.N;
}

// TMA coordinates (y, z) of query row r: maps [B*H][N][d], or token-major
// [total][H][d] for packed sequences.
template <class IT>
__device__ __forceinline__ void q_coords(const IT& I, int r, int& y, int& z) {
    if constexpr (is_packed<IT>()) { y = I.h; z = I.tb + r; }
    else { y = r; z = I.bh; }
}

// TMA coordinates of key / value row r.
template <class IT>
__device__ __forceinline__ void kv_coords(const IT& I, int r, const FwdParams& p, int& y, int& z) {
    if constexpr (is_packed<IT>()) { y = I.h / (p.H / p.Hkv); z = I.tbk + r; }
    else { y = r; z = I.kvh; }
}

// Row index of output row `row` (O has d elements per row) and of its LSE.
template <class IT>
__device__ __forceinline__ size_t out_row(const IT& I, int row, const FwdParams& p) {
    if constexpr (is_packed<IT>()) return (size_t)(I.tb + row) * p.H + I.h;
    else return (size_t)I.bh * p.N + row;
}
template <class IT>
__device__ __forceinline__ size_t lse_index(const IT& I, int row, const FwdParams& p) {
    if constexpr (is_packed<IT>())  // [H, total]; uniform lengths (no cu_seqlens): [B, H, N]
        return p.cu_seqlens ? (size_t)I.h * p.total + I.tb + row : ((size_t)I.b * p.H + I.h) * p.N + row;
    else return (size_t)I.bh * p.N + row;
}

// SPLITK: the kernel instance that also runs split-key units (compiled
// separately so that the plain forward carries none of their bookkeeping).
// VARLEN: the instance for packed variable-length sequences.
// WINDOW: the sliding-window instance (p is a FwdParamsWin).
// RECT: rectangular attention (p is a FwdParamsRect): Nk keys, causal offset coff.
template <class C, bool CAUSAL, bool SPLITK, bool VARLEN, bool WINDOW = false, bool SPARSE = false, bool RECT = false>
__device__ __forceinline__ ItemT<VARLEN, WINDOW, SPARSE> get_item(int unit, const ParamsT<WINDOW, SPARSE, RECT>& p) {
    ItemT<VARLEN, WINDOW, SPARSE> I;
    const int BH = p.B * p.H;
    int it = unit, s = 0, S = 1;
    I.part = -1;
    if (SPLITK && unit >= p.num_whole) {  // split unit: key range s of S of item `it`
        const int t = unit - p.num_whole;
        S = p.splits;
        it = p.num_whole + t / S;
        s = t % S;
        I.part = t;
    }
    int qp;
    fwd_item_coords(it, CAUSAL, BH, p.num_qp, I.bh, qp);
    dcheck(chk::tile_ok(I.bh, BH, qp, p.num_qp), kErrCheckTile);
    I.b = I.bh / p.H;
    const int h = I.bh - I.b * p.H;
    I.kvh = I.b * p.Hkv + h / (p.H / p.Hkv);
    int kvl, rows;
    if constexpr (VARLEN) {
        // no cu_seqlens: B sequences of N tokens each ([B, N, H, d] tensors)
        const int a = p.cu_seqlens ? __ldg(p.cu_seqlens + I.b) : I.b * p.N;
        const int e = p.cu_seqlens ? __ldg(p.cu_seqlens + I.b + 1) : a + p.N;
        I.h = h;
        I.tb = a;
        I.seqlen = max(0, min(e - a, p.N));
        kvl = rows = I.seqlen;
        I.tbk = a;
        I.coff = 0;
        if (p.cu_seqlens_k) {  // its own key range; causal: the queries are the last len_q positions
            I.tbk = __ldg(p.cu_seqlens_k + I.b);
            kvl = max(0, __ldg(p.cu_seqlens_k + I.b + 1) - I.tbk);
            I.coff = kvl - rows;
        }
    } else if constexpr (RECT) {
        rows = p.N;
        kvl = p.Nk;
        if (p.kv_lens) kvl = min(max(__ldg(p.kv_lens + I.b), 0), p.Nk);
    } else {
        kvl = rows = p.N;
        if (p.kv_lens) kvl = min(max(__ldg(p.kv_lens + I.b), 0), p.N);
    }
    I.kvl = kvl;
    I.row0 = qp * (C::QT * C::BR);
    I.nmax = 0;
    if constexpr (SPARSE) {
        // each tile's list, without the trailing blocks that hold no visible
        // key for any of its rows (beyond kv_len, or above the causal diagonal)
        const int nnz = __ldg(p.row_ptr + p.nqb);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int r0 = I.row0 + t * C::BR;
            int off = 0, cnt = 0;
            if (r0 < rows) {
                const int qb = r0 / C::BR;
                off = min(max(__ldg(p.row_ptr + qb), 0), nnz);
                cnt = min(max(min(__ldg(p.row_ptr + qb + 1), nnz) - off, 0), p.nkb);
                int lim = kvl;
                if (CAUSAL) lim = min(lim, min(r0 + C::BR, rows));
                while (cnt > 0 && __ldg(p.col_idx + off + cnt - 1) * C::BC >= lim) --cnt;
            }
            I.off[t] = off;
            I.n[t] = cnt;
        }
        BlockMerge mg = block_merge(I, p);
        int u = 0;
        bool a0, a1;
        while (mg.c0 < mg.n0 || mg.c1 < mg.n1) {
            mg.next(a0, a1);
            ++u;
        }
        I.nmax = u;
        I.j0 = 0;
    } else if constexpr (WINDOW) {
        // keys [lo, hi) cover every row of tile t: lo from its first row's left
        // edge, hi from its last row's right edge (and kv_len / causal)
        int lb[2], nb[2], J0 = 0x7fffffff, J1 = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int r0 = I.row0 + t * C::BR;
            lb[t] = 0;
            nb[t] = 0;
            if (r0 < rows) {
                const int rl = min(r0 + C::BR, rows) - 1;
                int hi = kvl;
                if (CAUSAL) hi = min(hi, rl + 1);
                if (p.win_right >= 0) hi = min(hi, rl + p.win_right + 1);
                const int lo = (p.win_left >= 0) ? max(0, r0 - p.win_left) : 0;
                if (hi > lo) {
                    lb[t] = lo / C::BC;
                    nb[t] = (hi + C::BC - 1) / C::BC - lb[t];
                    J0 = min(J0, lb[t]);
                    J1 = max(J1, lb[t] + nb[t]);
                }
            }
        }
        I.j0 = (J1 > 0) ? J0 : 0;
        I.nmax = (J1 > 0) ? J1 - J0 : 0;
        I.n[0] = nb[0];
        I.n[1] = nb[1];
        I.a[0] = nb[0] > 0 ? lb[0] - I.j0 : 0;
        I.a[1] = nb[1] > 0 ? lb[1] - I.j0 : 0;
    } else {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int r0 = I.row0 + t * C::BR;
            int n = 0;
            if (r0 < rows) {
                int cols = kvl;
                if constexpr (RECT) {
                    // the tile's largest query index (rows r0 .. rl, query = row % qmod)
                    const int rl = min(r0 + C::BR, rows) - 1;
                    const int qmax = (rl / p.qmod != r0 / p.qmod) ? p.qmod - 1 : rl % p.qmod;
                    if (CAUSAL) cols = min(cols, max(0, qmax + 1 + p.coff));
                } else if constexpr (VARLEN) {
                    if (CAUSAL) cols = min(cols, max(0, r0 + C::BR + I.coff));
                } else {
                    if (CAUSAL) cols = min(cols, r0 + C::BR);
                }
                n = (cols + C::BC - 1) / C::BC;
            }
            I.n[t] = n;
            I.nmax = max(I.nmax, n);
        }
        I.j0 = 0;
        if (SPLITK && S > 1) {
            const int j0 = (int)((long long)I.nmax * s / S), j1 = (int)((long long)I.nmax * (s + 1) / S);
            I.nmax = 0;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                I.n[t] = max(0, min(j1, I.n[t]) - j0);
                I.nmax = max(I.nmax, I.n[t]);
            }
            I.j0 = j0;
        }
    }
    return I;
}

// S_t = Q_t K^T over the head dimension (both operands K-major, 128B swizzle).
// With SPLIT, the three products hi.hi + hi.lo + lo.hi accumulate in turn.
// q_desc / k_desc: descriptors of the tile bases (hi parts); all per-MMA offsets
// are compile-time constants added to the start-address field.
template <class C>
__device__ __forceinline__ void issue_S(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
    if (elect_one()) {
#pragma unroll
        for (int part = 0; part < (C::SPLIT ? 3 : 1); ++part) {
            const uint64_t qd = desc_add(q_desc, part == 2 ? C::QT * C::Q_TILE : 0);
            const uint64_t kd = desc_add(k_desc, part == 1 ? C::KV_TILE : 0);
#pragma unroll
            for (int kk = 0; kk < C::S_STEPS; ++kk) {
                const uint32_t off_in = (kk % 4) * 32;
                const uint64_t a = desc_add(qd, (kk / 4) * C::Q_BOX + off_in);
                const uint64_t b = desc_add(kd, (kk / 4) * C::KV_BOX + off_in);
                const uint32_t acc = (part > 0 || kk > 0) ? 1u : 0u;
                if constexpr (C::FP8)
                    mma_f8_ss(d_tmem, a, b, C::IDESC_S, acc);
                else
                    mma_f16_ss(d_tmem, a, b, C::IDESC_S, acc);
            }
        }
    }
    __syncwarp();
}

// O_t (+)= P_t V over the keys; P_t from TMEM, V MN-major (head dim contiguous).
// KK0 / KK1: the range of K steps issued (the whole block by default).
template <class C, int KK0 = 0, int KK1 = C::PV_STEPS>
__device__ __forceinline__ void issue_PV(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, bool accumulate) {
    if (elect_one()) {
#pragma unroll
        for (int kk = KK0; kk < KK1; ++kk) {
            const uint64_t b = desc_add(v_desc, kk * C::KSTEP * 128);
            const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
            if constexpr (C::FP8)
                mma_f8_ts(o_tmem, p_tmem + kk * 8, b, C::IDESC_PV, acc);
            else
                mma_f16_ts(o_tmem, p_tmem + kk * 8, b, C::IDESC_PV, acc);
        }
    }
    __syncwarp();
}

// 2^x for a pair (MUFU ex2; 2^-inf = 0 exactly for masked scores)
__device__ __forceinline__ float2 exp2_pair(float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); }

// P = 2^(S * cm - m) for one row of a key block, written over the row's S
// columns in TMEM as the A operand of the P V product (bf16 pairs, or E4M3
// quadruples with the value-scale fold lg).  Returns the row sums: l (exact
// weights, divided by the fold) and, for FP8, lq (the E4M3-rounded weights).
// CH0 / CH1: the range of chunks (of CH columns) computed; the whole block by
// default.
template <class C, int CH0 = 0, int CH1 = -1>
__device__ __forceinline__ void exp_block(const float (&s)[C::BC], const float (&cm)[2], const float (&lg)[2],
                                          const float (&inv_w)[2], float mb, uint32_t tS, float& lsum,
                                          float& lqsum) {
    constexpr int CH = C::FP8 ? 64 : 32;  // columns per 16-word TMEM store
    constexpr int CHE = CH1 < 0 ? C::BC / CH : CH1;
    lsum = 0.f;
    lqsum = 0.f;
#pragma unroll
    for (int ch = CH0; ch < CHE; ++ch) {
        const int h = (ch * CH) / (C::BC / 2);
        const float2 cs2 = make_float2(cm[h], cm[h]), cb2 = make_float2(lg[h] - mb, lg[h] - mb);
        uint32_t w[16];
        float2 a2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if constexpr (C::FP8) {
            // lq sums the E4M3-rounded weights the P V product actually uses, so
            // O stays a convex combination of the value rows; l keeps the exact
            // sum for the LSE
            __half2 hacc = __float2half2_rn(0.f);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float* se = s + ch * CH + 4 * e;
                const float2 p01 = exp2_pair(ffma2(make_float2(se[0], se[1]), cs2, cb2));
                const float2 p23 = exp2_pair(ffma2(make_float2(se[2], se[3]), cs2, cb2));
                a2[e & 3] = fadd2(a2[e & 3], fadd2(p01, p23));
                w[e] = pack_e4m3x4(p01.x, p01.y, p23.x, p23.y);
                hacc = __hadd2(hacc, __hadd2(e4m3x2_to_half2(w[e] & 0xFFFFu), e4m3x2_to_half2(w[e] >> 16)));
            }
            const float2 hs = __half22float2(hacc);
            lqsum += (hs.x + hs.y) * inv_w[h];
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float2 pp = exp2_pair(ffma2(make_float2(s[ch * CH + 2 * e], s[ch * CH + 2 * e + 1]), cs2, cb2));
                a2[e & 3] = fadd2(a2[e & 3], pp);
                w[e] = pack_bf16x2(pp.x, pp.y);
            }
        }
        const float2 t2 = fadd2(fadd2(a2[0], a2[1]), fadd2(a2[2], a2[3]));
        lsum += (t2.x + t2.y) * inv_w[h];
        tmem_st16(tS + ch * 16, w);
    }
}

template <class C, bool OUT_F32>
__device__ __forceinline__ void store_row_chunk(void* o_row, int c0, const float (&v)[32]) {
    if constexpr (OUT_F32) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(o_row) + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(o_row) + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
    }
}

template <class C, bool CAUSAL, bool OUT_F32, bool SPLITK, bool VARLEN = false, bool WINDOW = false,
          bool SPARSE = false, bool RECT = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tql,
               const __grid_constant__ CUtensorMap tkl, const ParamsT<WINDOW, SPARSE, RECT> p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto BAR = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8 * i; };
    FA_CHECK_BIND(p.err);

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR(C::B_QFULL + t), 1);
            mbar_init(BAR(C::B_QEMPTY + t), 1);
        }
        for (int s = 0; s < C::KSTAGES; ++s) {
            mbar_init(BAR(C::B_KFULL + s), 1);
            mbar_init(BAR(C::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::VSTAGES; ++s) {
            mbar_init(BAR(C::B_VFULL + s), 1);
            mbar_init(BAR(C::B_VEMPTY + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(BAR(C::B_SFULL + t), 1);
            mbar_init(BAR(C::B_PFULL + t), 128);
            mbar_init(BAR(C::B_OFULL + t), 1);
            mbar_init(BAR(C::B_OEMPTY + t), 128);
            mbar_init(BAR(C::B_PHALF + t), 128);
        }
        mbar_init(BAR(C::B_DONE), 1);
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
            if (C::SPLIT) {
                prefetch_tmap(&tql);
                prefetch_tmap(&tkl);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // registers: the softmax warpgroups take what the producer / MMA warpgroup
    // (warps 8-11, 10 and 11 idle) does not need; 2 x 128 x C::REGS_SOFTMAX +
    // 128 x C::REGS_ISSUE equals the launch allocation of 384 x 168
    static_assert(2 * 128 * C::REGS_SOFTMAX + 128 * C::REGS_ISSUE <= kThreads * 168, "register split");

    if (warp >= 8) regs_dec<C::REGS_ISSUE>();
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp walks the schedule (so it stays converged); lane 0 issues.
        int kst = 0, vst = 0;
        uint32_t kph = 0, vph = 0, qe = 0;
        bool ok = true;
        for (int rd = 0; rd < snake_rounds(p.num_units) && ok; ++rd) {
            const int it = snake_item(rd, p.num_units);
            if (it < 0) continue;
            const auto I = get_item<C, CAUSAL, SPLITK, VARLEN, WINDOW, SPARSE, RECT>(it, p);
            if (I.nmax == 0) continue;
            // Q tile t of this item may load as soon as the previous item's last
            // S_t MMA has consumed the buffer (per-tile barriers), overlapping
            // the previous item's final P V products and epilogue
            for (int t = 0; t < C::QT && ok; ++t) {
                if (!(ok = wait_bounded_warp(BAR(C::B_QEMPTY + t), qe ^ 1, abort_flag, p.err, kErrWaitFwdProducer))) break;
                if (lane == 0) {
                    int y, z;
                    q_coords(I, I.row0 + t * C::BR, y, z);
                    mbar_arrive_expect_tx(BAR(C::B_QFULL + t), C::NPART * C::Q_TILE);
                    for (int part = 0; part < C::NPART; ++part)
                        for (int bx = 0; bx < C::NBOX; ++bx)
                            tma_load_3d(sbase + C::OFF_Q + (part * C::QT + t) * C::Q_TILE + bx * C::Q_BOX,
                                        part ? &tql : &tq, BAR(C::B_QFULL + t), bx * C::BOX_ELEMS, y, z);
                }
                __syncwarp();
            }
            if (!ok) break;
            qe ^= 1;
            // K runs one tile ahead of V (K_0 K_1 V_0 K_2 V_1 ...): S(j+1) needs K_{j+1}
            // before P V(j+1) needs V_{j+1}
            [[maybe_unused]] BlockMerge mg;
            [[maybe_unused]] int kb_cur = 0, kb_prev = 0;  // block-sparse: key blocks of the stream
            if constexpr (SPARSE) mg = block_merge(I, p);
            for (int idx = 0; idx <= I.nmax && ok; ++idx) {
                if constexpr (SPARSE) {
                    kb_prev = kb_cur;
                    if (idx < I.nmax) {
                        bool a0, a1;
                        kb_cur = mg.next(a0, a1);
                    }
                }
                if (idx < I.nmax) {
                    if (!(ok = wait_bounded_warp(BAR(C::B_KEMPTY + kst), kph ^ 1, abort_flag, p.err, kErrWaitFwdProducer))) break;
                    if (lane == 0) {
                        int y, z;
                        kv_coords(I, (SPARSE ? kb_cur : I.j0 + idx) * C::BC, p, y, z);
                        mbar_arrive_expect_tx(BAR(C::B_KFULL + kst), C::K_STAGE);
                        for (int part = 0; part < C::NPART; ++part)
                            for (int bx = 0; bx < C::NBOX; ++bx)
                                tma_load_3d(sbase + C::OFF_K + kst * C::K_STAGE + part * C::KV_TILE + bx * C::KV_BOX,
                                            part ? &tkl : &tk, BAR(C::B_KFULL + kst), bx * C::BOX_ELEMS, y, z);
                    }
                    __syncwarp();
                    if (++kst == C::KSTAGES) { kst = 0; kph ^= 1; }
                }
                if (idx >= 1) {
                    const int j = idx - 1;
                    if (!(ok = wait_bounded_warp(BAR(C::B_VEMPTY + vst), vph ^ 1, abort_flag, p.err, kErrWaitFwdProducer))) break;
                    if (lane == 0) {
                        int y, z;
                        kv_coords(I, (SPARSE ? kb_prev : I.j0 + j) * C::BC, p, y, z);
                        mbar_arrive_expect_tx(BAR(C::B_VFULL + vst), C::KV_TILE);
                        for (int bx = 0; bx < C::NBOX; ++bx)
                            tma_load_3d(sbase + C::OFF_V + vst * C::KV_TILE + bx * C::KV_BOX, &tv, BAR(C::B_VFULL + vst),
                                        bx * C::BOX_ELEMS, y, z);
                    }
                    __syncwarp();
                    if (++vst == C::VSTAGES) { vst = 0; vph ^= 1; }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the schedule and waits; one elected lane issues
        // each tcgen05 op.  Shared-memory descriptors are built once here and
        // advanced by constants, so the issue rate stays above the tensor rate.
        int kst = 0, vst = 0;
        uint32_t kph = 0, vph = 0, qph = 0;
        uint32_t pph[2] = {0, 0}, oeph[2] = {0, 0};
        const uint64_t q_desc0 = sdesc_sw128(sbase + C::OFF_Q, 16, 1024);
        const uint64_t k_desc0 = sdesc_sw128(sbase + C::OFF_K, 16, 1024);
        const uint64_t v_desc0 = sdesc_sw128(sbase + C::OFF_V, C::KV_BOX, 1024);
        auto q_desc = [&](int t) { return desc_add(q_desc0, t * C::Q_TILE); };
        auto k_desc = [&](int st) { return desc_add(k_desc0, st * C::K_STAGE); };
        auto v_desc = [&](int st) { return desc_add(v_desc0, st * C::KV_TILE); };
        auto tS = [&](int t) { return tmem + (t ? C::TM_S1 : C::TM_S0); };
        auto tO = [&](int t) { return tmem + (t ? C::TM_O1 : C::TM_O0); };
        bool ok = true;
        for (int rd = 0; rd < snake_rounds(p.num_units) && ok; ++rd) {
            const int it = snake_item(rd, p.num_units);
            if (it < 0) continue;
            const auto I = get_item<C, CAUSAL, SPLITK, VARLEN, WINDOW, SPARSE, RECT>(it, p);
            if (I.nmax == 0) continue;
            for (int t = 0; t < 2 && ok; ++t)
                ok = wait_bounded_warp(BAR(C::B_QFULL + t), qph, abort_flag, p.err, kErrWaitFwdMma);
            if (!ok) break;
            qph ^= 1;
            if (!(ok = wait_bounded_warp(BAR(C::B_KFULL + kst), kph, abort_flag, p.err, kErrWaitFwdMma))) break;
            tc_fence_after();
            if constexpr (SPARSE) {
                // union step u: P V for the tiles that compute block u, then S for
                // the tiles that compute block u + 1 (a tile may skip blocks)
                BlockMerge mg = block_merge(I, p);
                bool cu[2], nx[2];
                mg.next(cu[0], cu[1]);
                int sd[2] = {0, 0}, pd[2] = {0, 0};  // S / P V products issued per tile
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (cu[t]) {
                        issue_S<C>(tS(t), q_desc(t), k_desc(kst));
                        mma_commit_w(BAR(C::B_SFULL + t));
                        ++sd[t];
                    }
                    if (sd[t] == item_n(I, t)) mma_commit_w(BAR(C::B_QEMPTY + t));  // Q_t no longer needed
                }
                mma_commit_w(BAR(C::B_KEMPTY + kst));
                if (++kst == C::KSTAGES) { kst = 0; kph ^= 1; }
                for (int u = 0; u < I.nmax && ok; ++u) {
                    nx[0] = nx[1] = false;
                    if (u + 1 < I.nmax) mg.next(nx[0], nx[1]);
                    bool vw = false, kw = false;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (cu[t]) {
                            if (!(ok = wait_bounded_warp(BAR(C::B_PFULL + t), pph[t], abort_flag, p.err, kErrWaitFwdMma))) break;
                            pph[t] ^= 1;
                            if (pd[t] == 0) {
                                if (!(ok = wait_bounded_warp(BAR(C::B_OEMPTY + t), oeph[t] ^ 1, abort_flag, p.err, kErrWaitFwdMma))) break;
                                oeph[t] ^= 1;
                            }
                            if (!vw) {
                                if (!(ok = wait_bounded_warp(BAR(C::B_VFULL + vst), vph, abort_flag, p.err, kErrWaitFwdMma))) break;
                                vw = true;
                            }
                            tc_fence_after();
                            issue_PV<C>(tO(t), tS(t), v_desc(vst), pd[t] > 0);
                            if (++pd[t] == item_n(I, t)) mma_commit_w(BAR(C::B_OFULL + t));
                        }
                        if (nx[t]) {
                            if (!kw) {
                                if (!(ok = wait_bounded_warp(BAR(C::B_KFULL + kst), kph, abort_flag, p.err, kErrWaitFwdMma))) break;
                                kw = true;
                                tc_fence_after();
                            }
                            issue_S<C>(tS(t), q_desc(t), k_desc(kst));
                            mma_commit_w(BAR(C::B_SFULL + t));
                            if (++sd[t] == item_n(I, t)) mma_commit_w(BAR(C::B_QEMPTY + t));
                        }
                    }
                    if (!ok) break;
                    mma_commit_w(BAR(C::B_VEMPTY + vst));
                    if (++vst == C::VSTAGES) { vst = 0; vph ^= 1; }
                    if (kw) {
                        mma_commit_w(BAR(C::B_KEMPTY + kst));
                        if (++kst == C::KSTAGES) { kst = 0; kph ^= 1; }
                    }
                    cu[0] = nx[0];
                    cu[1] = nx[1];
                }
            } else {
                for (int t = 0; t < 2; ++t) {
                    if (item_a(I, t) == 0) {  // (a tile that starts later issues its first S in the loop)
                        if (item_n(I, t) > 0) {
                            issue_S<C>(tS(t), q_desc(t), k_desc(kst));
                            mma_commit_w(BAR(C::B_SFULL + t));
                        }
                        if (item_n(I, t) <= 1) mma_commit_w(BAR(C::B_QEMPTY + t));  // Q_t no longer needed
                    }
                }
                mma_commit_w(BAR(C::B_KEMPTY + kst));
                if (++kst == C::KSTAGES) { kst = 0; kph ^= 1; }
                for (int j = 0; j < I.nmax && ok; ++j) {
                    bool vw = false, kw = false;
                    for (int t = 0; t < 2; ++t) {
                        const int ta = item_a(I, t), te = ta + item_n(I, t);  // tile t: blocks [ta, te)
                        if (j < ta || j >= te) {
                            if (j + 1 == ta) {  // tile t starts with the next block: its first S
                                if (!kw) {
                                    if (!(ok = wait_bounded_warp(BAR(C::B_KFULL + kst), kph, abort_flag, p.err, kErrWaitFwdMma))) break;
                                    kw = true;
                                    tc_fence_after();
                                }
                                issue_S<C>(tS(t), q_desc(t), k_desc(kst));
                                mma_commit_w(BAR(C::B_SFULL + t));
                                if (te - ta == 1) mma_commit_w(BAR(C::B_QEMPTY + t));
                            }
                            continue;
                        }
                        // bf16: the first half of P V as soon as that half of P is in TMEM
                        if (!(ok = wait_bounded_warp(BAR((C::SPLITP ? C::B_PHALF : C::B_PFULL) + t), pph[t],
                                                     abort_flag, p.err, kErrWaitFwdMma)))
                            break;
                        if (j == ta) {
                            if (!(ok = wait_bounded_warp(BAR(C::B_OEMPTY + t), oeph[t] ^ 1, abort_flag, p.err, kErrWaitFwdMma))) break;
                            oeph[t] ^= 1;
                        }
                        if (!vw) {
                            if (!(ok = wait_bounded_warp(BAR(C::B_VFULL + vst), vph, abort_flag, p.err, kErrWaitFwdMma))) break;
                            vw = true;
                        }
                        tc_fence_after();
                        if constexpr (C::SPLITP) {
                            issue_PV<C, 0, C::PV_STEPS / 2>(tO(t), tS(t), v_desc(vst), j > ta);
                            if (!(ok = wait_bounded_warp(BAR(C::B_PFULL + t), pph[t], abort_flag, p.err, kErrWaitFwdMma)))
                                break;
                            tc_fence_after();
                            issue_PV<C, C::PV_STEPS / 2, C::PV_STEPS>(tO(t), tS(t), v_desc(vst), true);
                        } else {
                            issue_PV<C>(tO(t), tS(t), v_desc(vst), j > ta);
                        }
                        pph[t] ^= 1;
                        if (j == te - 1) {
                            mma_commit_w(BAR(C::B_OFULL + t));
                        } else {
                            if (!kw) {
                                if (!(ok = wait_bounded_warp(BAR(C::B_KFULL + kst), kph, abort_flag, p.err, kErrWaitFwdMma))) break;
                                kw = true;
                                tc_fence_after();
                            }
                            issue_S<C>(tS(t), q_desc(t), k_desc(kst));
                            mma_commit_w(BAR(C::B_SFULL + t));
                            if (j + 2 == te) mma_commit_w(BAR(C::B_QEMPTY + t));  // last S_t issued
                        }
                    }
                    if (!ok) break;
                    mma_commit_w(BAR(C::B_VEMPTY + vst));
                    if (++vst == C::VSTAGES) { vst = 0; vph ^= 1; }
                    if (kw) {
                        mma_commit_w(BAR(C::B_KEMPTY + kst));
                        if (++kst == C::KSTAGES) { kst = 0; kph ^= 1; }
                    }
                }
            }
            if (!ok) break;
        }
        // drain: every MMA this warp issued has completed before TMEM is freed
        mma_commit_w(BAR(C::B_DONE));
        wait_bounded_warp(BAR(C::B_DONE), 0, abort_flag, p.err, kErrWaitDrain);
    } else if (warp < 8) {
        // ------------------------------------------------------------ softmax
        regs_inc<C::REGS_SOFTMAX>();
        const int t = warp >> 2;
        const int wq = warp & 3;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + (t ? C::TM_S1 : C::TM_S0);
        const uint32_t tO = tmem + lane_off + (t ? C::TM_O1 : C::TM_O0);
        const int r_in = wq * 32 + lane;
        uint32_t sph = 0, oph = 0;
        for (int rd = 0; rd < snake_rounds(p.num_units); ++rd) {
            const int it = snake_item(rd, p.num_units);
            if (it < 0) continue;
            const auto I = get_item<C, CAUSAL, SPLITK, VARLEN, WINDOW, SPARSE, RECT>(it, p);
            const int n = item_n(I, t);
            const int tile_row0 = I.row0 + t * C::BR;
            const int row = tile_row0 + r_in;
            const int nrows = item_rows(I, p);
            const size_t row_idx = out_row(I, row, p);
            // destination of this row: O / LSE, or the unit's partial (split keys)
            const size_t prow = (size_t)I.part * 256 + t * C::BR + r_in;
            char* orow = reinterpret_cast<char*>(p.o) + row_idx * C::D * (OUT_F32 ? 4 : 2);
            float* lse_dst = (SPLITK && I.part >= 0)
                                 ? p.lse_part + prow
                                 : p.lse + lse_index(I, row, p);
            auto emit = [&](int c, const float (&f)[32]) {
                if (SPLITK && I.part >= 0) {
                    float4* dst = reinterpret_cast<float4*>(p.o_part + prow * C::D + c);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
                } else {
                    store_row_chunk<C, OUT_F32>(orow, c, f);
                }
            };
            if (n == 0) {
                if (row < nrows) {  // no visible key (kv_len = 0, or an empty key range): O = 0, LSE = -inf
                    float z[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
                    for (int c = 0; c < C::D; c += 32) emit(c, z);
                    *lse_dst = -INFINITY;
                }
                continue;
            }
            // FP8: per-row query scale and the head's largest value-block scale
            float sq_row = 1.f, sv_max = 1.f;
            if (C::FP8) {
                const float* svh = p.sv + (size_t)I.kvh * p.nblk;
                float mxs = 0.f;
                for (int i = lane; i < p.nblk; i += 32) mxs = fmaxf(mxs, __ldg(svh + i));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mxs = fmaxf(mxs, __shfl_xor_sync(0xffffffffu, mxs, o));
                sv_max = mxs;
                if (row < p.N) sq_row = __ldg(p.sq + (size_t)I.bh * p.nblk + row / 64);
            }
            float m = -INFINITY, l = 0.f;
            float lq = 0.f;  // FP8: sum of the E4M3-rounded weights (normalises O)
            const float w_scale = C::FP8 ? kFp8Fold / sv_max : 0.f;  // FP8: w = value-block scale * w_scale
            // FP8: key / value scales of the two 64-key halves of block j, read one
            // block ahead so that the global-memory latency stays off the step
            float skn[2] = {1.f, 1.f}, svn[2] = {1.f, 1.f};
            auto load_scales = [&](int jj) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int blk = (I.j0 + item_a(I, t) + jj) * 2 + h;
                    skn[h] = (blk < p.nblk) ? __ldg(p.sk + (size_t)I.kvh * p.nblk + blk) : 1.f;
                    svn[h] = (blk < p.nblk) ? __ldg(p.sv + (size_t)I.kvh * p.nblk + blk) : sv_max;
                }
            };
            if (C::FP8) load_scales(0);
            bool ok = true;
            for (int j = 0; j < n; ++j) {
                // multipliers of the raw scores (log2 domain) per 64-key half, formed
                // before the wait for S
                float cm[2], lg[2] = {0.f, 0.f}, inv_w[2] = {1.f, 1.f};
                if (C::FP8) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        cm[h] = p.scale_log2 * sq_row * skn[h];
                        const float w = svn[h] * w_scale;
                        lg[h] = __log2f(w);
                        inv_w[h] = __frcp_rn(w);
                    }
                    if (j + 1 < n) load_scales(j + 1);
                } else {
                    cm[0] = cm[1] = p.scale_log2;
                }
                if (!(ok = wait_bounded_warp(BAR(C::B_SFULL + t), sph, abort_flag, p.err, kErrWaitFwdSoftmax))) break;
                sph ^= 1;
                tc_fence_after();
                uint32_t sr[C::BC];
                if constexpr (C::BC == 128) {
                    tmem_ld128_wait(tS, sr);
                } else {
                    tmem_ld64_wait(tS, sr);
                }
                float s[C::BC];
#pragma unroll
                for (int c = 0; c < C::BC; ++c) s[c] = __uint_as_float(sr[c]);
                int col0 = (I.j0 + item_a(I, t) + j) * C::BC;
                if constexpr (SPARSE) col0 = __ldg(p.col_idx + (t ? I.off[1] : I.off[0]) + j) * C::BC;
                // causal limit of a row: its query index (+ the rectangular offset)
                int coff = 0, qmin = tile_row0, qrow = row;
                if constexpr (VARLEN) coff = I.coff;
                if constexpr (RECT) {
                    const int rl = tile_row0 + C::BR - 1;
                    coff = p.coff;
                    qmin = (rl / p.qmod != tile_row0 / p.qmod) ? 0 : tile_row0 % p.qmod;
                    qrow = row % p.qmod;
                }
                bool need_mask = (col0 + C::BC > I.kvl) || (CAUSAL && col0 + C::BC - 1 > qmin + coff);
                if constexpr (WINDOW)  // blocks crossing some row's window edge
                    need_mask = need_mask || (p.win_right >= 0 && col0 + C::BC - 1 > tile_row0 + p.win_right) ||
                                (p.win_left >= 0 && col0 < tile_row0 + C::BR - 1 - p.win_left);
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < C::BC; ++c) {
                        const int col = col0 + c;
                        bool off = col >= I.kvl || (CAUSAL && col > qrow + coff);
                        if constexpr (WINDOW)
                            off = off || (p.win_right >= 0 && col > row + p.win_right) ||
                                  (p.win_left >= 0 && col < row - p.win_left);
                        if (off) s[c] = -INFINITY;
                    }
                }
                // O *= f over the row (O holds the blocks whose P V has completed)
                auto rescale_o = [&](float f) {
#pragma unroll 1
                    for (int c = 0; c < C::D; c += 32) {
                        uint32_t ov[32];
                        tmem_ld32_wait(tO + c, ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
                        tmem_st32(tO + c, ov);
                    }
                    tmem_st_wait();
                };
                float lsum, lqsum;
                if constexpr (C::FP8) {
                    // reference max first (P <= 2^kFp8Slack must hold for the E4M3 fold)
                    const float mx2 = fmaxf(row_max<C::BC / 2>(s) * cm[0], row_max<C::BC / 2>(s + C::BC / 2) * cm[1]);
                    const bool need = mx2 > m + kFp8Slack;
                    float alpha = 1.f;
                    if (need) {
                        alpha = ex2_approx(m - mx2);  // 0 when m = -inf
                        m = mx2;
                        l *= alpha;
                        lq *= alpha;
                    }
                    if (j > 0 && __any_sync(0xffffffffu, need)) rescale_o(alpha);
                    const float mb = (m == -INFINITY) ? 0.f : m;
                    exp_block<C>(s, cm, lg, inv_w, mb, tS, lsum, lqsum);
                    l += lsum;
                    lq += lqsum;
                } else {  // bf16: split P hand-off
                    // the block's row max first; the reference moves (and O is
                    // rescaled: S(j) complete means P V(j-1) has completed) only
                    // when it grew by more than kRescaleSlack
                    const float mx = row_max<C::BC>(s) * cm[0];
                    if (j == 0) {
                        m = mx;
                    } else {
                        const bool need = mx > m + kRescaleSlack;
                        if (__any_sync(0xffffffffu, need)) {
                            float alpha = 1.f;
                            if (need) {
                                alpha = ex2_approx(m - mx);  // 0 when m = -inf
                                m = mx;
                                l *= alpha;
                            }
                            rescale_o(alpha);
                        }
                    }
                    const float mb = (m == -INFINITY) ? 0.f : m;
                    float lsum2;
                    constexpr int NCH = C::BC / 32;
                    // Blocks with and without masked entries take separate (identical)
                    // copies of the exponential loop: measured 2.7% faster at long_head
                    // causal than one call site shared by both
                    if (need_mask)
                        exp_block<C, 0, NCH / 2>(s, cm, lg, inv_w, mb, tS, lsum, lqsum);
                    else
                        exp_block<C, 0, NCH / 2>(s, cm, lg, inv_w, mb, tS, lsum, lqsum);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(BAR(C::B_PHALF + t));
                    if (need_mask)
                        exp_block<C, NCH / 2, NCH>(s, cm, lg, inv_w, mb, tS, lsum2, lqsum);
                    else
                        exp_block<C, NCH / 2, NCH>(s, cm, lg, inv_w, mb, tS, lsum2, lqsum);
                    l += lsum + lsum2;
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(BAR(C::B_PFULL + t));
            }
            if (!ok) break;
            if (!wait_bounded_warp(BAR(C::B_OFULL + t), oph, abort_flag, p.err, kErrWaitFwdSoftmax)) break;
            oph ^= 1;
            tc_fence_after();
            float inv = (l > 0.f) ? 1.f / l : 0.f;
            if (C::FP8) inv = (lq > 0.f) ? sv_max * (1.f / kFp8Fold) / lq : 0.f;
#pragma unroll 1
            for (int c = 0; c < C::D; c += 32) {
                uint32_t ov[32];
                tmem_ld32_wait(tO + c, ov);
                float f[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(ov[i]) * inv;
                if (row < nrows) emit(c, f);
            }
            tc_fence_before();
            mbar_arrive(BAR(C::B_OEMPTY + t));
            if (row < nrows) *lse_dst = (l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kProducerWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <class C, bool CAUSAL, bool OUT_F32, bool SPLITK = false, bool VARLEN = false, bool WINDOW = false,
          bool SPARSE = false, bool RECT = false>
cudaError_t launch(const FwdMaps& m, const ParamsT<WINDOW, SPARSE, RECT>& p, int grid, cudaStream_t stream) {
    auto kern = fwd_kernel<C, CAUSAL, OUT_F32, SPLITK, VARLEN, WINDOW, SPARSE, RECT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM, stream>>>(m.q, m.k, m.v, m.q_lo, m.k_lo, p);
    return cudaGetLastError();
}

// Rectangular attention (Nq != Nk), through the split-key instance.
template <class C>
cudaError_t launch_rect(bool causal, const FwdMaps& m, const FwdParamsRect& p, int grid, cudaStream_t s) {
    return causal ? launch<C, true, false, true, false, false, false, true>(m, p, grid, s)
                  : launch<C, false, false, true, false, false, false, true>(m, p, grid, s);
}

// Block-sparse (block lists of 128 x 128 blocks).
template <class C>
cudaError_t launch_sparse(bool causal, const FwdMaps& m, const FwdParamsSparse& p, int grid, cudaStream_t s) {
    return causal ? launch<C, true, false, false, false, false, true>(m, p, grid, s)
                  : launch<C, false, false, false, false, false, true>(m, p, grid, s);
}

// Sliding window (causal folded into the window's right edge by the caller).
template <class C>
cudaError_t launch_window(const FwdMaps& m, const FwdParamsWin& p, int grid, cudaStream_t s) {
    return launch<C, false, false, false, false, true>(m, p, grid, s);
}

template <class C>
cudaError_t launch_varlen_window(const FwdMaps& m, const FwdParamsWin& p, int grid, cudaStream_t s) {
    return launch<C, false, false, false, true, true>(m, p, grid, s);
}

template <class C>
cudaError_t launch_varlen(bool causal, const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
    return causal ? launch<C, true, false, false, true>(m, p, grid, s) : launch<C, false, false, false, true>(m, p, grid, s);
}

template <class C>
cudaError_t launch_splitk(bool causal, const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
    return causal ? launch<C, true, false, true>(m, p, grid, s) : launch<C, false, false, true>(m, p, grid, s);
}

template <class C>
cudaError_t launch_any(bool causal, bool out_f32, const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t s) {
    if (causal) return out_f32 ? launch<C, true, true>(m, p, grid, s) : launch<C, true, false>(m, p, grid, s);
    return out_f32 ? launch<C, false, true>(m, p, grid, s) : launch<C, false, false>(m, p, grid, s);
}

}  // namespace fwd
}  // namespace fa

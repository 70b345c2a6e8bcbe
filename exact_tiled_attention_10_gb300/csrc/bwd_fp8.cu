// FP8 backward of exact tiled attention for sm_103a (d = 128).
//
// What it computes is Algorithm 2 of the FA-v2 analysis page
// ("解析 FlashAttention（4）：FlashAttention-v2", §5.4), as the bf16 backward
// does, with the low-precision scheme chapter 18 §18.6.2 describes for the
// FlashAttention-3 backward: the products run on FP8 tensor cores, dS is
// quantised to E5M2 before the two products that consume it (dQ = dS K,
// dK = dS^T Q), and the gradients are accumulated in float32 (TMEM for dK,
// dV; the float32 dQ accumulator in global memory) and written as float32.
//
// Inputs are the FP8 forward's: Q8, K8, V8 (E4M3 codes with one scale per
// 64-row block, X ~= s_blk X8), its O (bf16) and LSE, and the upstream
// gradient dO, which the host quantises to E4M3 the same way (dO8, s_do):
// the gradients are those of the dequantised inputs under the dequantised
// upstream gradient dO^ = s_do dO8.
// Per step (one 128-key block j of the item x one 128-query block i):
//   S^T  = K8 Q8^T                (E4M3 x E4M3; s_k per key row, s_q per
//                                  64-query half folded into the softmax)
//   P    = exp(S - LSE)           (float32)
//   dV  += P''^T dO8              (P'' = E4M3(P s_do / max s_do * 448), from
//                                  TMEM; the dO block scale rides on P)
//   dP^T = V8 dO8^T               (E4M3 x E4M3; s_v s_do applied after)
//   dS   = P (dP - D)             (float32; D = rowsum(dO^ O), dO^ = s_do dO8,
//                                  the same dequantised gradient dP sees)
//   dK  += Xk^T Q8,  Xk = E5M2(dS s_q / max s_q * c)   (E5M2 x E4M3)
//   dQ^T = K8t Xq,   Xq = E5M2(dS s_k / max s_k * c)   (E4M3 x E5M2)
// where K8t is K8 transposed ([d][keys], written by the host's transpose
// kernel) and c a power of two per head that keeps |dS| c below the E5M2
// maximum: |dS| <= P |dP - D| <= 2.01 d max|dO| max|V| (O is a convex
// combination of the dequantised value rows, rounded to bf16).  Every scale
// that varies along a product's reduction dimension is folded into the
// operand that is quantised here, so each product has one constant factor,
// applied to its float32 result.
//
// GB300 mapping: the bf16 backward's persistent, warp-specialised design
// (bwd_kernel.cuh) with 128-query steps -- every FP8 operand row is then
// 128 bytes, one 128-byte swizzle row -- and one TMEM step slot:
//   TMEM: dV [0,128) | dK [128,256) | S^T [256,384) (P'' aliased, 32 columns)
//         | dP^T [384,512) (dQ^T aliased once dS is formed)
//   warps 0-7: two compute warpgroups (query halves), 8-11: dQ drain,
//   12: TMA producer, 13: MMA issue.
#include "common.cuh"
#include "ptx.cuh"

namespace fa {
namespace bwd8 {

constexpr int kThreads = 448;
constexpr int kDqWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int D = 128, BC = 128, BR = 128, HALF = 64;
constexpr int TILE = 128 * 128;  // one 128-row x 128-byte FP8 tile
constexpr int STAGES = 2;        // Q8 / dO8 ring
constexpr int TM_DV = 0, TM_DK = 128, TM_S = 256, TM_X = 384, TM_COLS = 512;
// shared memory map (tiles 1024-byte aligned)
constexpr int OFF_K = 0, OFF_V = TILE, OFF_KT = 2 * TILE;
constexpr int OFF_Q = 3 * TILE;
constexpr int OFF_DO = OFF_Q + STAGES * TILE;
constexpr int OFF_XK = OFF_DO + STAGES * TILE;
constexpr int OFF_XQ = OFF_XK + TILE;
constexpr int DQ_WARP_BYTES = 128 * 32 * 4;  // [128 queries][32 head-dim] float32
constexpr int OFF_DQ = OFF_XQ + TILE;
constexpr int STAT_BYTES = 2 * BR * 4;  // lse2[128], D[128]
constexpr int OFF_STAT = OFF_DQ + 4 * DQ_WARP_BYTES;
constexpr int OFF_BAR = OFF_STAT + STAGES * STAT_BYTES;
enum {
    B_KVFULL = 0, B_KVEMPTY, B_QFULL, B_QEMPTY = B_QFULL + STAGES, B_SFULL = B_QEMPTY + STAGES, B_DPFULL, B_PFULL,
    B_DSFULL, B_DSEMPTY, B_DQFULL, B_DQEMPTY, B_ACCFULL, B_ACCEMPTY, B_DONE, NBAR
};
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_MISC + 16 + 1024;
static_assert(SMEM <= 232448, "shared memory budget");
constexpr uint32_t IDESC_S = idesc_make(kFmtE4M3, kFmtE4M3, 0, 0, 128, 128);   // S^T, dP^T
constexpr uint32_t IDESC_DV = idesc_make(kFmtE4M3, kFmtE4M3, 0, 1, 128, 128);  // P''^T dO8
constexpr uint32_t IDESC_DK = idesc_make(kFmtE5M2, kFmtE4M3, 0, 1, 128, 128);  // Xk^T Q8
constexpr uint32_t IDESC_DQ = idesc_make(kFmtE4M3, kFmtE5M2, 0, 1, 128, 128);  // K8t Xq

struct Item {
    int bh, b, kt, kvl, i0, n;
};

__device__ __forceinline__ Item get_item(int it, const BwdFp8Params& p, bool causal) {
    Item I;
    const int BH = p.B * p.H;
    if (causal) {  // key blocks near the start see the most queries: first
        I.kt = it / BH;
        I.bh = it % BH;
    } else {
        I.bh = it / p.num_kt;
        I.kt = it % p.num_kt;
    }
    dcheck(chk::tile_ok(I.bh, BH, I.kt, p.num_kt), kErrCheckTile);
    I.b = I.bh / p.H;
    I.kvl = p.kv_lens ? min(max(__ldg(p.kv_lens + I.b), 0), p.N) : p.N;
    const int key0 = I.kt * BC;
    const int iend = (p.N + BR - 1) / BR;
    I.i0 = causal ? I.kt : 0;  // BR = BC: query block kt is the first that sees key block kt
    I.n = (key0 >= I.kvl) ? 0 : max(iend - I.i0, 0);
    return I;
}

// Largest block scale of one head (warp-wide; every lane gets the result).
__device__ __forceinline__ float head_max(const float* s, int nblk) {
    float m = 0.f;
    for (int i = threadIdx.x & 31; i < nblk; i += 32) m = fmaxf(m, __ldg(s + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m > 0.f ? m : 1.f;
}

// The per-head factors of one item: maxima of the block scales and the power
// of two c that keeps |dS| c below the E5M2 range.
struct HeadScales {
    float sq_max, sk_max, sv_max, sdo_max, c;
};
__device__ __forceinline__ HeadScales head_scales(const BwdFp8Params& p, int bh) {
    HeadScales h;
    const size_t o = (size_t)bh * p.nblk;
    h.sq_max = head_max(p.sq + o, p.nblk);
    h.sk_max = head_max(p.sk + o, p.nblk);
    h.sv_max = head_max(p.sv + o, p.nblk);
    h.sdo_max = head_max(p.sdo + o, p.nblk);
    const float bound = 2.01f * D * (448.f * h.sdo_max) * (448.f * h.sv_max);
    h.c = exp2f(floorf(log2f(49152.f / bound)));
    return h;
}

__device__ __forceinline__ float blk_scale(const float* s, int bh, int nblk, int row) {
    const int blk = row / 64;
    return blk < nblk ? __ldg(s + (size_t)bh * nblk + blk) : 0.f;
}

// 448 threads = 14 warps, 4 of them on two of the SM's four sub-partitions,
// whose register files hold 16384 registers each: at most 128 a thread.
__global__ void __launch_bounds__(kThreads, 1)
    bwd_fp8_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tkt, const __grid_constant__ CUtensorMap tdq,
                   const BwdFp8Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool causal = p.causal != 0;
    auto BAR = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8 * i; };
    FA_CHECK_BIND(p.err);

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_KVFULL), 1);
        mbar_init(BAR(B_KVEMPTY), 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(BAR(B_QFULL + s), 1);
            mbar_init(BAR(B_QEMPTY + s), 1);
        }
        mbar_init(BAR(B_SFULL), 1);
        mbar_init(BAR(B_DPFULL), 1);
        mbar_init(BAR(B_PFULL), 256);
        mbar_init(BAR(B_DSFULL), 256);
        mbar_init(BAR(B_DSEMPTY), 1);
        mbar_init(BAR(B_DQFULL), 1);
        mbar_init(BAR(B_DQEMPTY), 128);
        mbar_init(BAR(B_ACCFULL), 1);
        mbar_init(BAR(B_ACCEMPTY), 256);
        mbar_init(BAR(B_DONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp) {
        tmem_alloc(smem_u32(tmem_slot), TM_COLS);
        tmem_relinquish();
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            prefetch_tmap(&tdo);
            prefetch_tmap(&tkt);
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
            const Item I = get_item(it, p, causal);
            if (I.n == 0) continue;
            if (!(ok = wait_bounded_warp(BAR(B_KVEMPTY), kve ^ 1, abort_flag, p.err, kErrWaitBwdProducer))) break;
            kve ^= 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(BAR(B_KVFULL), 3 * TILE);
                tma_load_3d(sbase + OFF_K, &tk, BAR(B_KVFULL), 0, I.kt * BC, I.bh);
                tma_load_3d(sbase + OFF_V, &tv, BAR(B_KVFULL), 0, I.kt * BC, I.bh);
                tma_load_3d(sbase + OFF_KT, &tkt, BAR(B_KVFULL), I.kt * BC, 0, I.bh);
            }
            __syncwarp();
            for (int s = 0; s < I.n; ++s) {
                const int i = I.i0 + s;
                if (!(ok = wait_bounded_warp(BAR(B_QEMPTY + st), ph ^ 1, abort_flag, p.err, kErrWaitBwdProducer))) break;
                if (lane == 0) {
                    const uint32_t bar = BAR(B_QFULL + st);
                    mbar_arrive_expect_tx(bar, 2 * TILE + STAT_BYTES);
                    tma_load_3d(sbase + OFF_Q + st * TILE, &tq, bar, 0, i * BR, I.bh);
                    tma_load_3d(sbase + OFF_DO + st * TILE, &tdo, bar, 0, i * BR, I.bh);
                    const size_t roff = (size_t)I.bh * p.Np + (size_t)i * BR;
                    bulk_load(sbase + OFF_STAT + st * STAT_BYTES, p.lse2 + roff, BR * 4, bar);
                    bulk_load(sbase + OFF_STAT + st * STAT_BYTES + BR * 4, p.dvec + roff, BR * 4, bar);
                }
                __syncwarp();
                if (++st == STAGES) { st = 0; ph ^= 1; }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // step s: [dP(s) once dQ(s-1) is drained] | dV(s) | S(s+1) | dK(s), dQ(s)
        int st = 0, st_ahead = 0;
        uint32_t qph_ahead = 0, kvph = 0, aeph = 0, pph = 0, dsph = 0, dqeph = 0;
        const uint64_t k_kd = sdesc_sw128(sbase + OFF_K, 16, 1024);
        const uint64_t v_kd = sdesc_sw128(sbase + OFF_V, 16, 1024);
        const uint64_t kt_kd = sdesc_sw128(sbase + OFF_KT, 16, 1024);
        const uint64_t q_kd0 = sdesc_sw128(sbase + OFF_Q, 16, 1024);
        const uint64_t q_mn0 = sdesc_sw128(sbase + OFF_Q, TILE, 1024);
        const uint64_t do_kd0 = sdesc_sw128(sbase + OFF_DO, 16, 1024);
        const uint64_t do_mn0 = sdesc_sw128(sbase + OFF_DO, TILE, 1024);
        const uint64_t xk_kd = sdesc_sw128(sbase + OFF_XK, 16, 1024);
        const uint64_t xq_mn = sdesc_sw128(sbase + OFF_XQ, TILE, 1024);
        bool ok = true;
        bool dq_pending = false;  // a dQ^T tile sits in the dP^T columns until drained
        auto open_step = [&]() -> bool {  // S^T of the next step into the S columns
            if (!wait_bounded_warp(BAR(B_QFULL + st_ahead), qph_ahead, abort_flag, p.err, kErrWaitBwdMma)) return false;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f8_ss(tmem + TM_S, desc_add(k_kd, kk * 32), desc_add(q_kd0, st_ahead * TILE + kk * 32), IDESC_S,
                              kk > 0);
            }
            __syncwarp();
            mma_commit_w(BAR(B_SFULL));
            if (++st_ahead == STAGES) { st_ahead = 0; qph_ahead ^= 1; }
            return true;
        };
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item(it, p, causal);
            if (I.n == 0) continue;
            if (!(ok = wait_bounded_warp(BAR(B_KVFULL), kvph, abort_flag, p.err, kErrWaitBwdMma))) break;
            kvph ^= 1;
            if (!(ok = open_step())) break;
            for (int s = 0; s < I.n; ++s) {
                // dP^T(s), once the previous dQ^T has left the columns
                if (dq_pending) {  // phase k of DQEMPTY completes when the k-th dQ^T tile is drained
                    if (!(ok = wait_bounded_warp(BAR(B_DQEMPTY), dqeph, abort_flag, p.err, kErrWaitBwdMma))) break;
                    dqeph ^= 1;
                    dq_pending = false;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f8_ss(tmem + TM_X, desc_add(v_kd, kk * 32), desc_add(do_kd0, st * TILE + kk * 32), IDESC_S,
                                  kk > 0);
                }
                __syncwarp();
                mma_commit_w(BAR(B_DPFULL));
                // dV(s) += P''^T dO8
                if (!(ok = wait_bounded_warp(BAR(B_PFULL), pph, abort_flag, p.err, kErrWaitBwdMma))) break;
                pph ^= 1;
                if (s == 0) {
                    if (!(ok = wait_bounded_warp(BAR(B_ACCEMPTY), aeph ^ 1, abort_flag, p.err, kErrWaitBwdMma))) break;
                    aeph ^= 1;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f8_ts(tmem + TM_DV, tmem + TM_S + (kk >> 1) * HALF + (kk & 1) * 8,
                                  desc_add(do_mn0, st * TILE + kk * 32 * 128), IDESC_DV, (s > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
                // S^T(s+1): the S columns (P'') are read by dV(s), issued before
                if (s + 1 < I.n && !(ok = open_step())) break;
                // dK(s), dQ^T(s)
                if (!(ok = wait_bounded_warp(BAR(B_DSFULL), dsph, abort_flag, p.err, kErrWaitBwdMma))) break;
                dsph ^= 1;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f8_ss(tmem + TM_DK, desc_add(xk_kd, kk * 32), desc_add(q_mn0, st * TILE + kk * 32 * 128),
                                  IDESC_DK, (s > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
                mma_commit_w(BAR(B_QEMPTY + st));
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f8_ss(tmem + TM_X, desc_add(kt_kd, kk * 32), desc_add(xq_mn, kk * 32 * 128), IDESC_DQ,
                                  kk > 0);
                }
                __syncwarp();
                mma_commit_w(BAR(B_DQFULL));
                mma_commit_w(BAR(B_DSEMPTY));
                dq_pending = true;
                if (++st == STAGES) st = 0;
            }
            if (!ok) break;
            mma_commit_w(BAR(B_KVEMPTY));
            mma_commit_w(BAR(B_ACCFULL));
        }
        mma_commit_w(BAR(B_DONE));
        wait_bounded_warp(BAR(B_DONE), 0, abort_flag, p.err, kErrWaitDrain);
    } else if (warp < 8) {
        // ------------------------------------------------------------ compute warpgroups
        const int h = warp >> 2;  // query half of every step
        const int wq = warp & 3;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const int kr = wq * 32 + lane;  // key row of this thread within the block
        int st = 0;
        uint32_t qph = 0, acph = 0, sph = 0, dpph = 0, dseph = 0;
        bool ok = true;
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item(it, p, causal);
            const int key = I.kt * BC + kr;
            const size_t krow = (size_t)I.bh * p.N + key;
            if (I.n == 0) {  // no query sees the key block: zero gradients for its keys
                if (key < p.N) {
                    float4* dst = reinterpret_cast<float4*>(h ? p.dk : p.dv) + krow * (D / 4);
#pragma unroll 4
                    for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                continue;
            }
            const HeadScales hs = head_scales(p, I.bh);
            const float sk_row = blk_scale(p.sk, I.bh, p.nblk, key);
            const float sv_row = blk_scale(p.sv, I.bh, p.nblk, key);
            const bool key_ok = key < I.kvl;
            for (int s = 0; s < I.n; ++s) {
                const int i = I.i0 + s;
                const int q0 = i * BR + h * HALF;  // first query of this half
                // this half's 64 queries are one 64-row block of Q and of dO
                const float sq = blk_scale(p.sq, I.bh, p.nblk, q0);
                const float sdo = blk_scale(p.sdo, I.bh, p.nblk, q0);
                if (!(ok = wait_bounded_warp(BAR(B_QFULL + st), qph, abort_flag, p.err, kErrWaitBwdCompute))) break;
                const float* lse2 = reinterpret_cast<const float*>(smem + OFF_STAT + st * STAT_BYTES) + h * HALF;
                const float* dvec = lse2 + BR;
                if (!(ok = wait_bounded_warp(BAR(B_SFULL), sph, abort_flag, p.err, kErrWaitBwdCompute))) break;
                sph ^= 1;
                tc_fence_after();
                uint32_t sr[HALF];
                tmem_ld64_wait(tmem + lane_off + TM_S + h * HALF, sr);
                const bool need_mask = (I.kt * BC + BC > I.kvl) || (causal && I.kt * BC + BC - 1 > i * BR);
                const float cmul = p.scale_log2 * sk_row * sq;
                float pv[HALF];
#pragma unroll
                for (int c = 0; c < HALF; c += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
                    pv[c + 0] = ex2_approx(fmaf(__uint_as_float(sr[c + 0]), cmul, -l4.x));
                    pv[c + 1] = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), cmul, -l4.y));
                    pv[c + 2] = ex2_approx(fmaf(__uint_as_float(sr[c + 2]), cmul, -l4.z));
                    pv[c + 3] = ex2_approx(fmaf(__uint_as_float(sr[c + 3]), cmul, -l4.w));
                }
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < HALF; ++c)
                        if (!key_ok || (causal && key > q0 + c)) pv[c] = 0.f;
                }
                // P'' = E4M3(P s_do / max s_do * 448) over this half's S columns
                {
                    const float pw = sdo / hs.sdo_max * 448.f;
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_e4m3x4(pv[4 * e] * pw, pv[4 * e + 1] * pw, pv[4 * e + 2] * pw, pv[4 * e + 3] * pw);
                    tmem_st16(tmem + lane_off + TM_S + h * HALF, w);
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(BAR(B_PFULL));
                // dS = P (dP - D), as the two E5M2 operands
                if (!(ok = wait_bounded_warp(BAR(B_DPFULL), dpph, abort_flag, p.err, kErrWaitBwdCompute))) break;
                dpph ^= 1;
                tc_fence_after();
                if (!(ok = wait_bounded_warp(BAR(B_DSEMPTY), dseph ^ 1, abort_flag, p.err, kErrWaitBwdCompute))) break;
                dseph ^= 1;
                const float dpm = sv_row * sdo;
                const float kmul = sq / hs.sq_max * hs.c, qmul = sk_row / hs.sk_max * hs.c;
                uint8_t* xk_row = smem + OFF_XK + kr * 128;
                uint8_t* xq_row = smem + OFF_XQ + kr * 128;
#pragma unroll
                for (int cc = 0; cc < HALF; cc += 32) {
                    uint32_t dr[32];
                    tmem_ld32_wait(tmem + lane_off + TM_X + h * HALF + cc, dr);
#pragma unroll
                    for (int c16 = 0; c16 < 32; c16 += 16) {
                        const int c = cc + c16;
                        float ds[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) ds[e] = pv[c + e] * fmaf(__uint_as_float(dr[c16 + e]), dpm, -dvec[c + e]);
                        uint4 wk, wq4;
                        wk.x = pack_e5m2x4(ds[0] * kmul, ds[1] * kmul, ds[2] * kmul, ds[3] * kmul);
                        wk.y = pack_e5m2x4(ds[4] * kmul, ds[5] * kmul, ds[6] * kmul, ds[7] * kmul);
                        wk.z = pack_e5m2x4(ds[8] * kmul, ds[9] * kmul, ds[10] * kmul, ds[11] * kmul);
                        wk.w = pack_e5m2x4(ds[12] * kmul, ds[13] * kmul, ds[14] * kmul, ds[15] * kmul);
                        wq4.x = pack_e5m2x4(ds[0] * qmul, ds[1] * qmul, ds[2] * qmul, ds[3] * qmul);
                        wq4.y = pack_e5m2x4(ds[4] * qmul, ds[5] * qmul, ds[6] * qmul, ds[7] * qmul);
                        wq4.z = pack_e5m2x4(ds[8] * qmul, ds[9] * qmul, ds[10] * qmul, ds[11] * qmul);
                        wq4.w = pack_e5m2x4(ds[12] * qmul, ds[13] * qmul, ds[14] * qmul, ds[15] * qmul);
                        // 16-byte chunk (h * 64 + c) / 16 of the row, in the 128-byte swizzle
                        const int chunk = (h * HALF + c) / 16;
                        if (dcheck(chk::range_ok(kr * 128 + ((chunk ^ (kr & 7)) * 16), 16, TILE), kErrCheckSmem)) {
                            *reinterpret_cast<uint4*>(xk_row + ((chunk ^ (kr & 7)) * 16)) = wk;
                            *reinterpret_cast<uint4*>(xq_row + ((chunk ^ (kr & 7)) * 16)) = wq4;
                        }
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(BAR(B_DSFULL));
                if (++st == STAGES) { st = 0; qph ^= 1; }
            }
            if (!ok) break;
            // epilogue: warpgroup 0 writes dV, warpgroup 1 dK (float32)
            if (!(ok = wait_bounded_warp(BAR(B_ACCFULL), acph, abort_flag, p.err, kErrWaitBwdCompute))) break;
            acph ^= 1;
            tc_fence_after();
            const float mul = h ? p.scale * hs.sq_max / hs.c : hs.sdo_max / 448.f;
            float* dst = reinterpret_cast<float*>(h ? p.dk : p.dv) + krow * D;
            const uint32_t tacc = tmem + lane_off + (h ? TM_DK : TM_DV);
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t a[32];
                tmem_ld32_wait(tacc + c, a);
                if (key < p.N) {
                    float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d4[e] = make_float4(__uint_as_float(a[4 * e]) * mul, __uint_as_float(a[4 * e + 1]) * mul,
                                            __uint_as_float(a[4 * e + 2]) * mul, __uint_as_float(a[4 * e + 3]) * mul);
                }
            }
            tc_fence_before();
            mbar_arrive(BAR(B_ACCEMPTY));
        }
    } else if (warp < 12) {
        // ------------------------------------------------------------ dQ drain warps
        // lane = head-dim row (wq * 32 + lane) of dQ^T, columns = the step's 128 queries
        const int wq = warp - kDqWarp0;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t stage = sbase + OFF_DQ + wq * DQ_WARP_BYTES;
        float* stage_f = reinterpret_cast<float*>(smem + OFF_DQ + wq * DQ_WARP_BYTES);
        uint32_t dqph = 0;
        bool ok = true;
        for (int rd = 0; rd < snake_rounds(p.num_items) && ok; ++rd) {
            const int it = snake_item(rd, p.num_items);
            if (it < 0) continue;
            const Item I = get_item(it, p, causal);
            if (I.n == 0) continue;
            const HeadScales hs = head_scales(p, I.bh);
            const float mul = hs.sk_max / hs.c;  // the conversion applies `scale`
            for (int s = 0; s < I.n; ++s) {
                const int i = I.i0 + s;
                if (!(ok = wait_bounded_warp(BAR(B_DQFULL), dqph, abort_flag, p.err, kErrWaitBwdDq))) break;
                dqph ^= 1;
                tc_fence_after();
                // half 0 staged, half 1 loaded, the columns released, half 1 staged
                if (lane == 0) bulk_wait_group_read<0>();  // the previous reduction has read the staging
                __syncwarp();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[64];
                    tmem_ld64_wait(tmem + lane_off + TM_X + half * 64, v);
                    if (half == 1) {
                        tc_fence_before();
                        mbar_arrive(BAR(B_DQEMPTY));
                    }
                    if (dcheck(chk::range_ok(((half * 64 + 63) * 32 + lane) * 4, 4, DQ_WARP_BYTES), kErrCheckSmem))
#pragma unroll
                        for (int q = 0; q < 64; ++q) stage_f[(half * 64 + q) * 32 + lane] = __uint_as_float(v[q]) * mul;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_2d(&tdq, stage, wq * 32, I.bh * p.Np + i * BR);
                    bulk_commit_group();
                }
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
        tmem_dealloc(tmem, TM_COLS);
    }
}

// K8 [B*H][N][128] -> K8t [B*H][128][Np] (keys >= N zero): one 128-key x
// 128-column tile per CTA iteration through shared memory; each thread then
// writes 4 consecutive keys of one head-dim row as one 32-bit word.
__global__ void __launch_bounds__(256) transpose_k8_kernel(const uint8_t* __restrict__ k8, uint8_t* __restrict__ kt,
                                                           int BH, int N, int Np) {
    __shared__ uint8_t tile[128][132];
    const int ntile = Np / 128;
    for (long t = blockIdx.x; t < (long)BH * ntile; t += gridDim.x) {
        const int bh = (int)(t / ntile), k0 = (int)(t % ntile) * 128;
        __syncthreads();
        for (int j = threadIdx.x; j < 128 * 8; j += 256) {  // 16-byte chunks: key j / 8, columns 16 (j % 8)
            const int key = j / 8, c = (j % 8) * 16;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (k0 + key < N) v = __ldg(reinterpret_cast<const uint4*>(k8 + ((size_t)bh * N + k0 + key) * 128 + c));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) *reinterpret_cast<uint32_t*>(&tile[key][c + 4 * e]) = w[e];
        }
        __syncthreads();
        for (int w = threadIdx.x; w < 128 * 32; w += 256) {  // word w: head-dim row w / 32, keys 4 (w % 32) ..
            const int dr = w / 32, kk = (w % 32) * 4;
            const uint32_t word = (uint32_t)tile[kk][dr] | ((uint32_t)tile[kk + 1][dr] << 8) |
                                  ((uint32_t)tile[kk + 2][dr] << 16) | ((uint32_t)tile[kk + 3][dr] << 24);
            *reinterpret_cast<uint32_t*>(kt + ((size_t)bh * 128 + dr) * Np + k0 + kk) = word;
        }
    }
}

}  // namespace bwd8

cudaError_t launch_bwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                           const CUtensorMap& tkt, const CUtensorMap& tdq, const BwdFp8Params& p, int grid,
                           cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd8::bwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bwd8::SMEM);
    if (e != cudaSuccess) return e;
    bwd8::bwd_fp8_kernel<<<grid, bwd8::kThreads, bwd8::SMEM, stream>>>(tq, tk, tv, tdo, tkt, tdq, p);
    return cudaGetLastError();
}

cudaError_t launch_transpose_k8(const void* k8, void* kt, int BH, int N, int Np, int grid, cudaStream_t stream) {
    bwd8::transpose_k8_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint8_t*>(k8),
                                                        reinterpret_cast<uint8_t*>(kt), BH, N, Np);
    return cudaGetLastError();
}

}  // namespace fa

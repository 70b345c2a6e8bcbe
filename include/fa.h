/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact tiled attention library.
 *
 * Exact multi-head attention O = softmax(scale * Q K^T + M) V computed tile by
 * tile: the forward keeps a per-row online-softmax state and writes only O and
 * the per-row log-sum-exp; the backward rebuilds each probability tile from
 * that log-sum-exp.  Sources (titles of the pages the method is taken from):
 *   [FA2]  "解析 FlashAttention（4）：FlashAttention-v2" -- §4 Algorithm 1
 *          (forward), §5.2 (D = rowsum(dO*O)), §5.4 Algorithm 2 (backward).
 *   [WIKI] "分块 Attention：重建概率，累计梯度" -- §01 running state, §04
 *          gradients with 1/sqrt(d) on dQ and dK, fully-masked-row convention.
 *   [CH18] "第18章 FlashAttention" -- §18.2.2 causal mask M_ij = -inf for
 *          j > i and the padding (column) mask of Table 18-3; §18.6.2 FP8
 *          E4M3 with per-block scale s = max|X| / 448; §18.7.1 API
 *          (softmax_scale defaults to 1/sqrt(headdim), causal in-kernel);
 *          §18.8.2 FlashDecoding (split key sequence, merged partials).
 *
 * Common conventions for every entry point
 * ----------------------------------------
 *  * Tensors are DEVICE pointers owned by the caller, contiguous row-major:
 *      q, k, v, o, dout, dq, dk, dv : [B, H, N, d]
 *      lse                          : [B, H, N] float32, natural log of the
 *                                     scaled scores; -inf on a fully masked row
 *      kv_lens                      : [B] int32 on the device, or NULL (= N).
 *    Every pointer must be 16-byte aligned (TMA requirement).
 *  * Masking: key j is visible to query i iff j < kv_lens[b] and, when
 *    causal != 0, j <= i (top-left aligned, N_q = N_k).  kv_lens[b] outside
 *    [0, N] is clamped to that range.  A query row with no visible key gets
 *    O = 0, LSE = -inf and zero gradients ([WIKI] §04).
 *  * scale multiplies Q K^T; pass 1/sqrt(d) for standard attention.
 *  * d must be 64 or 128 (bf16 paths); 128 for the FP8 path.  N >= 1.
 *  * Calls are asynchronous on `stream` and never synchronise.  Argument
 *    errors are detected on the host and returned before any launch; launch
 *    failures return FA_ERR_CUDA.  Faults detected inside a kernel (a
 *    pipeline wait that exceeded its time limit) set a device error word that
 *    fa_check_device_status() reports as FA_ERR_TIMEOUT.
 *  * The library allocates no device memory.  Scratch memory is passed in by
 *    the caller as `workspace` (sizes from the *_workspace_size queries).
 *  * On any non-OK status, fa_last_error() returns a message (thread-local).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, ... */
    FA_ERR_UNSUPPORTED = 2, /* head dim / dtype / device not supported        */
    FA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed            */
    FA_ERR_TIMEOUT = 4      /* a kernel gave up waiting (device error word)    */
} fa_status;

typedef enum { FA_BF16 = 0, FA_F32 = 1 } fa_dtype;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* fa_stream_t;

/* Library version, (major << 16) | minor. */
int fa_version(void);

/* Thread-local description of the last non-OK status ("" if none). */
const char* fa_last_error(void);

/* Waits for `stream`, then reads and clears the device error word.  Returns
 * FA_ERR_TIMEOUT if a kernel recorded a timed-out pipeline wait since the last
 * call, FA_ERR_CUDA if the stream itself reports an error, else FA_OK. */
fa_status fa_check_device_status(fa_stream_t stream);

/* Failure-detection self-test: launches one warp that waits, through the same
 * bounded pipeline wait the kernels use, on a barrier nothing ever arrives
 * on.  It gives up after limit_us microseconds (1 .. 1e6), writes 0 to the
 * device int *waited_out (1 would mean the wait completed), sets the device
 * error word, and returns; the next fa_check_device_status() then reports
 * FA_ERR_TIMEOUT and clears the word.  No trap, no hang, no fault. */
fa_status fa_selftest_wait_timeout(unsigned int limit_us, int* waited_out, fa_stream_t stream);

/* Self-test of the E4M3 quantiser's division (fa_quantize_fp8 divides every
 * element of a 64-row block by the block's scale s = amax / 448, [CH18]
 * §18.6.2): for n float32 device elements, q_fast[i] = x[i] / s[i % ns] by
 * the quantiser's shared-divisor method and q_ieee[i] = the IEEE float32
 * quotient; the two must agree bit for bit.  Device pointers; asynchronous on
 * `stream`. */
fa_status fa_selftest_quantiser_division(const float* x, const float* s, int ns, size_t n,
                                         float* q_fast, float* q_ieee, fa_stream_t stream);

/* ---------------------------------------------------------------- forward */

/* bf16 forward ([FA2] §4 Algorithm 1).  q,k,v: bf16 inputs; o: bf16 output;
 * lse: float32 [B,H,N].  Tiles of 128 query rows x 128 keys (64 keys when
 * N <= 128). */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 const int* kv_lens, fa_stream_t stream);

/* Extended forward.
 *   dtype   FA_BF16: as fa_fwd.  FA_F32: q,k,v,o are float32.  q and k are
 *           split into bf16 high and low parts (x = hi + lo, ~16 significant
 *           bits) in `workspace` and the scores are formed from three bf16
 *           tensor-core products, hi.hi + hi.lo + lo.hi, with float32
 *           accumulation; v and the probabilities enter P V as bf16; O is
 *           written as float32.
 *   block_c 0 = automatic, or 64 / 128 keys per tile (FA_F32 with d = 128
 *           needs 64).
 *   workspace, workspace_bytes: at least fa_fwd_workspace_size(dtype,...)
 *           bytes of device memory (NULL allowed when that size is 0). */
size_t fa_fwd_workspace_size(fa_dtype dtype, int B, int H, int N, int d);
fa_status fa_fwd_ex(fa_dtype dtype, int block_c, const void* q, const void* k, const void* v,
                    void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
                    const int* kv_lens, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/* Split-key forward, bf16 ([CH18] §18.8.2, FlashDecoding: the key sequence of
 * a query block is cut into contiguous ranges computed by separate thread
 * blocks, and the per-range results are merged with the online-softmax
 * weights).  Same inputs, outputs and semantics as fa_fwd; the work units
 * are (head, 256 query rows, key range) and a second kernel merges the
 * ranges: LSE = log sum_t exp(LSE_t), O = sum_t exp(LSE_t - LSE) O_t, where
 * O_t and LSE_t are the normalised output and LSE of range t (equivalent to
 * the chapter's merge of (m_t, l_t, unnormalised O_t), since
 * l_t exp(m_t) = exp(LSE_t)).
 *   num_splits  0: automatic -- whole items fill the full rounds of the
 *               persistent grid and only the remainder is split (2..4 ranges)
 *               when that shortens the last round; never for causal or
 *               key-padded calls (their items are unequal).  1: no split
 *               (exactly fa_fwd).  >= 2: every item in that many ranges (at
 *               most 64).
 *   workspace   device scratch for the partial results, at least
 *               fa_fwd_split_workspace_size(...) bytes, 16-byte aligned (NULL
 *               allowed when that size is 0).  FA_ERR_INVALID_ARG if smaller.
 * The plan depends on the current device's SM count; fa_fwd_split_count
 * returns the number of ranges the call will use (1 = not split). */
size_t fa_fwd_split_workspace_size(int B, int H, int N, int d, int causal, int has_kv_lens,
                                   int num_splits);
int fa_fwd_split_count(int B, int H, int N, int d, int causal, int has_kv_lens, int num_splits);
fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                       int num_splits, void* workspace, size_t workspace_bytes,
                       fa_stream_t stream);

/* Rectangular attention, bf16: Nq queries against Nk keys -- a decoding step
 * against a key/value cache (FlashDecoding, [CH18] §18.8.2: the query is
 * [b, n_q, d] with n_q << n_kv) or cross-attention.  q, o: [B,H,Nq,d]; k, v:
 * [B,Hkv,Nk,d]; lse [B,H,Nq]; kv_lens [B] (valid cache length per batch
 * item, clamped to [0, Nk]) or NULL.  With causal the queries are the last
 * Nq positions: query i sees keys j <= i + Nk - Nq.  Runs the split-key
 * form: num_splits = 0 plans the split (every item is cut into key ranges
 * when the items fill less than half the GPU), 1 = unsplit, >= 2 = that
 * many ranges per item (capped at 64).  Workspace:
 * fa_fwd_rect_workspace_size(...) bytes (0 when unsplit);
 * fa_fwd_rect_split_count gives the ranges per item the call will use.  The
 * query rows of the H / Hkv heads sharing a key/value head are processed as
 * one block of rows (they are contiguous in q), so each K / V tile is read
 * once per group. */
size_t fa_fwd_rect_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits);
int fa_fwd_rect_split_count(int B, int H, int Hkv, int Nq, int Nk, int d, int num_splits);
fa_status fa_fwd_rect(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                      const int* kv_lens, int num_splits, void* workspace, size_t workspace_bytes,
                      fa_stream_t stream);

/* Backward of the rectangular forward (cross-attention training; Nq query
 * rows, Nk keys, same causal reading), bf16: dq [B,H,Nq,d]; dk, dv
 * [B,Hkv,Nk,d] summed over the query heads sharing a key/value head; o and
 * lse from fa_fwd_rect.  Workspace: fa_bwd_rect_workspace_size(...) bytes
 * (at least fa_bwd_workspace_size(FA_BF16, B, H, Nq, d); the extra space
 * lets few key blocks split their query heads, as fa_bwd_gqa). */
size_t fa_bwd_rect_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d);
fa_status fa_bwd_rect(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                      const int* kv_lens, void* workspace, size_t workspace_bytes,
                      fa_stream_t stream);

/* Shared key/value heads (grouped-query attention; multi-query for Hkv = 1),
 * bf16.  q, o: [B,H,N,d]; k, v: [B,Hkv,N,d] with H a multiple of Hkv; query
 * head h attends with key/value head h / (H / Hkv) -- the head broadcast of
 * flash_attn_func API ([CH18] §18.7.1: with fewer key/value heads than query
 * heads, K and V are broadcast over the head dimension).  Otherwise as
 * fa_fwd.  FA_ERR_INVALID_ARG if H % Hkv != 0. */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Hkv, int N, int d, float scale, int causal,
                     const int* kv_lens, fa_stream_t stream);

/* Sliding-window attention (flash_attn_func's window_size = (left, right),
 * [CH18] §18.7.1; the block-skipping form of [CH18] §18.8.1), bf16, shapes
 * as fa_fwd_gqa (Hkv = H for ordinary multi-head attention): key j is
 * visible to query i only if i - window_left <= j <= i + window_right, -1
 * meaning no bound on that side, on top of the causal (j <= i) and key
 * padding masks.  Key blocks entirely outside a query tile's window are not
 * loaded or multiplied.  A row with no visible key gets O = 0, LSE = -inf.
 * FA_ERR_INVALID_ARG for an edge below -1; window (-1, -1) is fa_fwd_gqa. */
fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int Hkv, int N, int d, float scale, int causal,
                        int window_left, int window_right, const int* kv_lens,
                        fa_stream_t stream);

/* Block-sparse attention ([CH18] §18.8.1: per query block the list of key
 * blocks to compute; the others are neither loaded nor multiplied), bf16,
 * shapes as fa_fwd_gqa.  Blocks are 128 x 128: query block i (rows
 * 128 i .. 128 i + 127) attends to the keys of the key blocks
 * col_idx[row_ptr[i] .. row_ptr[i+1]-1] only, on top of the causal and key
 * padding masks; the same lists serve every batch item and head.
 * row_ptr: device int32 [nb + 1], nb = ceil(N / 128), non-decreasing, with
 * row_ptr[nb] = the number of entries of col_idx; col_idx: device int32,
 * each list ascending without repeats, entries in [0, nb).  The kernels
 * clamp list bounds to [0, row_ptr[nb]] but do not otherwise validate the
 * lists (malformed lists give wrong results).  A query block with an empty
 * list gets O = 0, LSE = -inf. */
fa_status fa_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Hkv, int N, int d, float scale, int causal,
                              const int* row_ptr, const int* col_idx, const int* kv_lens,
                              fa_stream_t stream);

/* Packed variable-length sequences (flash_attn_varlen_func, [CH18] §18.7.1),
 * bf16: sequence b holds tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 of the
 * token-major tensors q, o [total, H, d] and k, v [total, Hkv, d] (Hkv = H
 * for ordinary multi-head attention); there is no attention across
 * sequences and causal means key <= query within a sequence.  cu_seqlens:
 * device int32 [batch + 1], non-decreasing, cu_seqlens[0] = 0 and
 * cu_seqlens[batch] = total; max_seqlen >= every length (longer sequences
 * are cut to max_seqlen).  lse: float32 [H, total].  A sequence of length 0
 * produces nothing. */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens, int batch, int total, int max_seqlen, int H, int Hkv,
                        int d, float scale, int causal, fa_stream_t stream);

/* Packed sequences under a sliding window (flash_attn_varlen_func's
 * window_size, [CH18] §18.7.1): fa_fwd_varlen / fa_bwd_varlen with the window
 * of fa_fwd_window applied within each sequence (positions counted from the
 * sequence's first token; -1 = unbounded; causal = right edge at 0).  The
 * backward takes fa_bwd_varlen's workspace, or with deterministic != 0
 * fa_bwd_varlen_deterministic_workspace_size's (bitwise-repeatable results,
 * see fa_bwd_window_deterministic).  Not combined with separate key ranges
 * (FA_ERR_UNSUPPORTED). */
fa_status fa_fwd_varlen_window(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int* cu_seqlens, int batch, int total, int max_seqlen, int H,
                               int Hkv, int d, float scale, int causal, int window_left,
                               int window_right, fa_stream_t stream);
fa_status fa_bwd_varlen_window(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               const int* cu_seqlens, int batch, int total, int max_seqlen, int H,
                               int Hkv, int d, float scale, int causal, int window_left,
                               int window_right, int deterministic, void* workspace,
                               size_t workspace_bytes, fa_stream_t stream);

/* Packed sequences with their own key ranges (flash_attn_varlen_func's
 * cu_seqlens_q / cu_seqlens_k, [CH18] §18.7.1), bf16: sequence b has queries
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q, o [total_q, H, d] and keys
 * cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k, v [total_k, Hkv, d]; lse
 * float32 [H, total_q].  With causal, the queries of a sequence are its last
 * len_q positions: query i sees keys j <= i + len_k - len_q (as in
 * fa_fwd_rect); a query that sees no key gets O = 0, LSE = -inf.
 * max_seqlen_q >= every query length (longer sequences are cut); key
 * lengths are taken as given.  Same results as fa_fwd_rect on each sequence
 * alone. */
fa_status fa_fwd_varlen_kv(const void* q, const void* k, const void* v, void* o, float* lse,
                           const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                           int total_q, int total_k, int max_seqlen_q, int H, int Hkv, int d,
                           float scale, int causal, fa_stream_t stream);

/* Forward on flash_attn_func's own layout ([CH18] §18.7.1: q is (batch,
 * seqlen, nheads, headdim), k and v (batch, seqlen_k, nheads_k, headdim)),
 * bf16: q, o [B, N, H, d]; k, v [B, N, Hkv, d]; lse float32 [B, H, N].  Same
 * results as fa_fwd_gqa on the transposed tensors (no key padding: use
 * fa_fwd_varlen for sequences of different lengths); the kernels read the
 * rows in place through token-major tensor maps, with no transposition pass.
 * B * N must fit in 32 bits. */
fa_status fa_fwd_bnhd(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int N, int H, int Hkv, int d, float scale, int causal,
                      fa_stream_t stream);

/* --------------------------------------------------------------- backward */

/* Scratch for fa_bwd / fa_bwd_ex, in bytes: the row statistics
 * LSE*log2(e) and D = rowsum(dO*O) ([FA2] §5.2), 2 x [B,H,Np] float32, plus
 * the float32 dQ accumulator [B,H,Np,d] (Np = N rounded up to a multiple of
 * 128), plus, for FA_F32, bf16 copies of q, k, v, o and dout. */
size_t fa_bwd_workspace_size(fa_dtype dtype, int B, int H, int N, int d);

/* bf16 backward of L = sum(O * dout) ([FA2] §5.4 Algorithm 2; [WIKI] §04):
 * given q, k, v, the forward's o and lse and the upstream gradient dout,
 * writes dq, dk, dv (bf16, overwritten, not accumulated).  Launches three
 * kernels on `stream`: preprocess (D and zeroed dQ accumulator), the main
 * kernel parallel over key blocks, and the dQ conversion. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dout, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Deterministic backward (flash_attn_func's `deterministic` flag, chapter 18
 * §18.7.1): the same results as fa_bwd_gqa (Hkv = H: fa_bwd), but dq, dk
 * and dv are bitwise identical from run to run.  In fa_bwd, the key blocks
 * add their dQ parts into one float32 accumulator in whatever order they
 * finish, so the rounding differs between runs.  Here key block kt writes
 * float32 accumulator kt % A (A = 1 .. 8, from the shape: B, Hkv, N).  Each
 * quarter of a dQ tile of accumulator a takes its key blocks in increasing
 * order: the first stores, the others add.  A key block waits (bounded;
 * FA_ERR_TIMEOUT through fa_check_device_status) for the quarter's turn
 * counter.  A last kernel sums the A accumulators in order.  Key blocks that
 * run at the same time use different accumulators, so they seldom wait.
 * dq [B,H,N,d]; dk, dv [B,Hkv,N,d], summed over the query heads sharing a
 * key/value head; H % Hkv == 0.  The workspace needs
 * fa_bwd_deterministic_workspace_size(B, H, Hkv, N, d) bytes: fa_bwd's
 * layout, A - 1 more accumulators and the counters (zeroed by the call).
 * The kernel's CTAs (one per SM at most) wait on one another, so they must
 * all be resident: do not overlap two of these calls on one device.  A wait
 * that runs out ends the kernel with FA_ERR_TIMEOUT; it never hangs. */
size_t fa_bwd_deterministic_workspace_size(int B, int H, int Hkv, int N, int d);
fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               int B, int H, int Hkv, int N, int d, float scale, int causal,
                               const int* kv_lens, void* workspace, size_t workspace_bytes,
                               fa_stream_t stream);

/* Backward with shared key/value heads (see fa_fwd_gqa), bf16: dq is
 * [B,H,N,d]; dk, dv are [B,Hkv,N,d] and hold the sum over the H / Hkv query
 * heads that share each key/value head (the gradient of the broadcast).
 * Workspace: at least fa_bwd_workspace_size(FA_BF16, B, H, N, d) bytes.
 * With fa_bwd_gqa_workspace_size(B, H, Hkv, N, d) bytes (larger when there
 * are fewer than 2 x SMs key blocks in all), each key block's query heads
 * are split over several work units that write float32 partial dK / dV to
 * the extra space, summed by one more kernel: the causal longest-first
 * schedule then stays balanced.  fa_bwd_window uses the same extra space. */
size_t fa_bwd_gqa_workspace_size(int B, int H, int Hkv, int N, int d);
fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     int B, int H, int Hkv, int N, int d, float scale, int causal,
                     const int* kv_lens, void* workspace, size_t workspace_bytes,
                     fa_stream_t stream);

/* Backward of fa_fwd_window (same window and masks), bf16: dq [B,H,N,d];
 * dk, dv [B,Hkv,N,d] summed over the query heads sharing a key/value head.
 * Only query blocks inside some key's window are visited per key block.
 * Workspace: fa_bwd_workspace_size(FA_BF16, B, H, N, d). */
fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int B, int H, int Hkv, int N, int d, float scale, int causal,
                        int window_left, int window_right, const int* kv_lens,
                        void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Backward of fa_fwd_block_sparse (same lists and masks), bf16: dq
 * [B,H,N,d]; dk, dv [B,Hkv,N,d] summed over the query heads sharing a
 * key/value head.  A one-CTA kernel first transposes the lists into the
 * workspace (for every key block, its query blocks); each key block then
 * visits only those.  Workspace: fa_bwd_block_sparse_workspace_size(B, H, N,
 * d) bytes (fa_bwd_workspace_size plus the transposed lists).
 * FA_ERR_UNSUPPORTED beyond 12000 blocks (N > 1,536,000). */
size_t fa_bwd_block_sparse_workspace_size(int B, int H, int N, int d);
fa_status fa_bwd_block_sparse(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int N, int d, float scale, int causal,
                              const int* row_ptr, const int* col_idx, const int* kv_lens,
                              void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Backward of fa_fwd_varlen (packed variable-length sequences, bf16): dq
 * [total, H, d], dk, dv [total, Hkv, d] (summed over the query heads sharing
 * a key/value head), same cu_seqlens / max_seqlen / lse as the forward.
 * Workspace: fa_bwd_varlen_workspace_size(batch, max_seqlen, H, d) bytes --
 * LSE*log2(e) and D per (head, sequence) padded to 128 rows, 2 x
 * [H][batch][Np] float32, and the float32 dQ accumulator [H][batch][Np][d]
 * (Np = max_seqlen rounded up to 128). */
size_t fa_bwd_varlen_workspace_size(int batch, int max_seqlen, int H, int d);
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        const int* cu_seqlens, int batch, int total, int max_seqlen, int H,
                        int Hkv, int d, float scale, int causal, void* workspace,
                        size_t workspace_bytes, fa_stream_t stream);

/* Backward of fa_fwd_varlen_kv, bf16: dq [total_q, H, d]; dk, dv [total_k,
 * Hkv, d] (summed over the query heads sharing a key/value head).
 * deterministic != 0 gives bitwise-repeatable results (see
 * fa_bwd_deterministic).  max_seqlen_k >= every key length.  Workspace:
 * fa_bwd_varlen_kv_workspace_size(..., deterministic) bytes. */
size_t fa_bwd_varlen_kv_workspace_size(int batch, int max_seqlen_q, int max_seqlen_k, int H, int Hkv,
                                       int d, int deterministic);
fa_status fa_bwd_varlen_kv(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                           const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                           int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                           int Hkv, int d, float scale, int causal, int deterministic,
                           void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Backward of fa_fwd_bnhd, bf16: dq [B, N, H, d]; dk, dv [B, N, Hkv, d]
 * (summed over the query heads sharing a key/value head); o, lse, dout as
 * the forward wrote / read them.  Workspace:
 * fa_bwd_bnhd_workspace_size(B, N, H, d) bytes (the statistics and the
 * float32 dQ accumulator per (head, sequence), as for fa_bwd_varlen). */
size_t fa_bwd_bnhd_workspace_size(int B, int N, int H, int d);
fa_status fa_bwd_bnhd(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      int B, int N, int H, int Hkv, int d, float scale, int causal,
                      void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Deterministic versions of fa_bwd_varlen and fa_bwd_bnhd (the
 * `deterministic` flag of flash_attn_varlen_func / flash_attn_func,
 * [CH18] §18.7.1): same arguments and results, with dq, dk and dv bitwise
 * identical from run to run.  The fixed order, the A float32 accumulators
 * and the turn counters are those of fa_bwd_deterministic, per (head,
 * sequence) row group; A comes from (batch, Hkv, max_seqlen).  Workspace: the
 * *_deterministic_workspace_size bytes (the packed layout, A - 1 more
 * accumulators, the counters).  The same residency note as
 * fa_bwd_deterministic applies: do not overlap two of these calls on one
 * device. */
size_t fa_bwd_varlen_deterministic_workspace_size(int batch, int max_seqlen, int H, int Hkv, int d);
fa_status fa_bwd_varlen_deterministic(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, const int* cu_seqlens, int batch, int total,
                                      int max_seqlen, int H, int Hkv, int d, float scale,
                                      int causal, void* workspace, size_t workspace_bytes,
                                      fa_stream_t stream);
size_t fa_bwd_bnhd_deterministic_workspace_size(int B, int N, int H, int Hkv, int d);
fa_status fa_bwd_bnhd_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                    int B, int N, int H, int Hkv, int d, float scale, int causal,
                                    void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Deterministic versions of fa_bwd_window, fa_bwd_block_sparse and
 * fa_bwd_rect (same arguments and results).  The key blocks that visit a
 * query block take the accumulators in their order among that block's
 * visitors: under a sliding window they form a range that may start above
 * 0; with block lists they are the query block's list, the causal and
 * key-length cuts dropping only its tail (found by a binary search in
 * col_idx).  Workspace: fa_bwd_deterministic_workspace_size(B, H, Hkv, N, d)
 * for the window, the *_deterministic_workspace_size queries for the others
 * (block lists: plus their transposition, as for fa_bwd_block_sparse). */
fa_status fa_bwd_window_deterministic(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, int B, int H, int Hkv, int N, int d, float scale,
                                      int causal, int window_left, int window_right,
                                      const int* kv_lens, void* workspace, size_t workspace_bytes,
                                      fa_stream_t stream);
size_t fa_bwd_block_sparse_deterministic_workspace_size(int B, int H, int Hkv, int N, int d);
fa_status fa_bwd_block_sparse_deterministic(const void* q, const void* k, const void* v,
                                            const void* o, const float* lse, const void* dout,
                                            void* dq, void* dk, void* dv, int B, int H, int Hkv,
                                            int N, int d, float scale, int causal,
                                            const int* row_ptr, const int* col_idx,
                                            const int* kv_lens, void* workspace,
                                            size_t workspace_bytes, fa_stream_t stream);
size_t fa_bwd_rect_deterministic_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d);
fa_status fa_bwd_rect_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                    int B, int H, int Hkv, int Nq, int Nk, int d, float scale,
                                    int causal, const int* kv_lens, void* workspace,
                                    size_t workspace_bytes, fa_stream_t stream);

/* The three phases fa_bwd runs, callable one by one (bf16 tensors, same
 * workspace).  fa_bwd == fa_bwd_preprocess; fa_bwd_main; fa_bwd_dq.
 *   fa_bwd_preprocess: D = rowsum(dout * o) ([FA2] §5.2), LSE * log2(e) and
 *                      a zeroed float32 dQ accumulator, into `workspace`.
 *   fa_bwd_main:       the key-block-parallel kernel ([FA2] §5.4): writes
 *                      dk, dv and accumulates unscaled dQ into `workspace`.
 *   fa_bwd_dq:         dq = scale * accumulator, as bf16.
 * Each phase reads what the previous one wrote; call them in this order on
 * one stream (or order the streams). */
fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H, int N,
                            int d, void* workspace, size_t workspace_bytes, fa_stream_t stream);
fa_status fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk,
                      void* dv, int B, int H, int N, int d, float scale, int causal,
                      const int* kv_lens, void* workspace, size_t workspace_bytes,
                      fa_stream_t stream);
fa_status fa_bwd_dq(void* dq, int B, int H, int N, int d, float scale, void* workspace,
                    size_t workspace_bytes, fa_stream_t stream);

/* As fa_bwd with an element type: FA_F32 takes float32 q,k,v,o,dout and writes
 * float32 dq,dk,dv (the tensor cores see bf16-rounded copies). */
fa_status fa_bwd_ex(fa_dtype dtype, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                    int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                    void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Allocation-free backward (the pages have no counterpart: it only changes
 * where the scratch lives).  For callers that cannot allocate device memory,
 * e.g. a plugin inside a framework that owns the whole device-memory pool, or
 * a runtime that forbids allocation after start-up.  Same arguments and
 * results as fa_bwd, minus the workspace: the scratch is a fixed 128 MiB array
 * of device memory defined in this library, which every GPU that loads the
 * library keeps until the process exits.
 *   - Problems whose scratch (fa_bwd_workspace_size(FA_BF16, ...)) exceeds
 *     fa_bwd_noalloc_max_scratch() bytes are rejected with FA_ERR_INVALID_ARG.
 *   - The first call on each device looks up the array's device address (no
 *     allocation); make that first call before any stream capture.
 *   - Every call uses the same array and leaves its contents behind; each call
 *     re-initialises what it reads, but calls that overlap on the GPU (e.g. on
 *     two streams) race on it and must be serialised by the caller.
 *   - Calls no cudaMalloc / cudaFree and no allocating library routine. */
size_t fa_bwd_noalloc_max_scratch(void);
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal,
                         const int* kv_lens, fa_stream_t stream);

/* -------------------------------------------------------------------- FP8 */

/* Number of 64-row scale blocks per (b,h): ceil(N / 64). */
int fa_fp8_num_blocks(int N);

/* Per-block E4M3 quantisation ([CH18] §18.6.2).  For each (b, h) and each
 * block of 64 consecutive rows x all d columns: amax = max|x|, s = amax / 448
 * (s = 1 when amax = 0), x8 = E4M3(x / s) with round-to-nearest-even and
 * saturation to +-448 (division and rounding in float32).
 *   x_bf16: bf16 [B,H,N,d]; x_e4m3: uint8 [B,H,N,d]; scales: float32
 *   [B,H,fa_fp8_num_blocks(N)]. */
fa_status fa_quantize_fp8(const void* x_bf16, void* x_e4m3, float* scales,
                          int B, int H, int N, int d, fa_stream_t stream);

/* fa_quantize_fp8 of q [B,H,N,d], k and v [B,Hkv,N,d] in one launch (the
 * three inputs of fa_fwd_fp8 / fa_fwd_fp8_split), same codes and scales as
 * three separate calls: sq [B,H,ceil(N/64)], sk, sv [B,Hkv,ceil(N/64)].
 * FA_ERR_INVALID_ARG if H % Hkv != 0. */
fa_status fa_quantize_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8,
                              void* v8, float* sq, float* sk, float* sv, int B, int H, int Hkv,
                              int N, int d, fa_stream_t stream);

/* FP8 forward: q8/k8/v8 are E4M3 [B,H,N,d] with per-64-row-block scales
 * sq/sk/sv (as written by fa_quantize_fp8), so that X ~= s_block * X8.
 * S = scale * (s_q s_k) (Q8 K8^T) accumulates in float32; the softmax runs in
 * float32; the probabilities are re-quantised to E4M3 (with the value scale of
 * each key block folded in) for the P V product; O is written as bf16 and LSE
 * as float32.  d must be 128. */
fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8,
                     const float* sq, const float* sk, const float* sv,
                     void* o, float* lse, int B, int H, int N, int d, float scale,
                     int causal, const int* kv_lens, fa_stream_t stream);

/* FP8 forward with shared key/value heads (see fa_fwd_gqa): q8, sq for H
 * query heads; k8, v8 [B,Hkv,N,d] and sk, sv [B,Hkv,ceil(N/64)] for Hkv key /
 * value heads, as fa_quantize_fp8_qkv writes them; H % Hkv == 0. */
fa_status fa_fwd_fp8_gqa(const void* q8, const void* k8, const void* v8,
                         const float* sq, const float* sk, const float* sv,
                         void* o, float* lse, int B, int H, int Hkv, int N, int d, float scale,
                         int causal, const int* kv_lens, fa_stream_t stream);

/* Split-key FP8 forward: fa_fwd_fp8 with the key ranges and merge of
 * fa_fwd_split (same num_splits and workspace rules; d = 128). */
fa_status fa_fwd_fp8_split(const void* q8, const void* k8, const void* v8,
                           const float* sq, const float* sk, const float* sv,
                           void* o, float* lse, int B, int H, int N, int d, float scale,
                           int causal, const int* kv_lens, int num_splits, void* workspace,
                           size_t workspace_bytes, fa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */

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
 *  * One call per pass: fa_attn_fwd / fa_attn_bwd take an fa_attn_params
 *    block that names the layout, the masks, the head sharing and the options
 *    of every variant, and one validation routine accepts or refuses the
 *    combination before any launch.  fa_fwd, fa_bwd, fa_quantize_fp8 and
 *    fa_fwd_fp8 are the plain calls of the method (bf16 / E4M3 tensors
 *    [B,H,N,d]); they run the same code as the parameter-block calls.
 *  * On any non-OK status, fa_last_error() returns a message (thread-local).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

/* Symbols of this header are the library's exported interface; everything
 * else in the shared library is built with hidden visibility. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, ... */
    FA_ERR_UNSUPPORTED = 2, /* head dim / dtype / device not supported        */
    FA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed            */
    FA_ERR_TIMEOUT = 4,     /* a kernel gave up waiting (device error word)    */
    FA_ERR_CHECK = 5        /* checked build (FA_DEBUG): an access broke a rule */
} fa_status;

/* Element type of the attention tensors.  FA_E4M3: q, k, v are E4M3 codes
 * (uint8) with per-64-row-block float32 scales (fa_quantize_fp8), o and dout
 * are bf16, dq / dk / dv are float32 (see fa_attn_bwd). */
typedef enum { FA_BF16 = 0, FA_F32 = 1, FA_E4M3 = 2 } fa_dtype;

/* Tensor layouts of fa_attn_params.
 *   FA_LAYOUT_BHND   q, o, dout, dq [B, H, N_q, d]; k, v, dk, dv [B, Hkv, N_k, d];
 *                    lse [B, H, N_q].
 *   FA_LAYOUT_BNHD   flash_attn_func's own layout ([CH18] §18.7.1: q is
 *                    (batch, seqlen, nheads, headdim)): q, o, dout, dq
 *                    [B, N, H, d]; k, v, dk, dv [B, N, Hkv, d]; lse [B, H, N];
 *                    read in place, no transposition pass.  B * N < 2^31.
 *   FA_LAYOUT_PACKED flash_attn_varlen_func ([CH18] §18.7.1): sequences of
 *                    unequal length concatenated token by token; q, o, dout,
 *                    dq [total_q, H, d]; k, v, dk, dv [total_k, Hkv, d]; lse
 *                    float32 [H, total_q]; sequence b holds query tokens
 *                    cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key tokens
 *                    cu_seqlens_k[b] .. (cu_seqlens_k NULL: the same
 *                    ranges); no attention across sequences. */
typedef enum { FA_LAYOUT_BHND = 0, FA_LAYOUT_BNHD = 1, FA_LAYOUT_PACKED = 2 } fa_layout;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* fa_stream_t;

/* Library version, (major << 16) | minor. */
FA_API int fa_version(void);

/* Thread-local description of the last non-OK status ("" if none). */
FA_API const char* fa_last_error(void);

/* Waits for `stream`, then reads and clears the device error word.  Returns
 * FA_ERR_CHECK if, in the checked build (compiled with FA_DEBUG=1, shipped as
 * libfa_gb300_debug.so), a kernel found an access that breaks one of its
 * rules -- a TMA coordinate or alignment, a TMEM lane quadrant or column
 * range, a shared-memory tile store out of its tile, a work item decoded out
 * of range -- and skipped it; else FA_ERR_TIMEOUT if a kernel recorded a
 * timed-out pipeline wait since the last call; FA_ERR_CUDA if the stream
 * itself reports an error; else FA_OK. */
FA_API fa_status fa_check_device_status(fa_stream_t stream);

/* Failure-detection self-test: launches one warp that waits, through the same
 * bounded pipeline wait the kernels use, on a barrier nothing ever arrives
 * on.  It gives up after limit_us microseconds (1 .. 1e6), writes 0 to the
 * device int *waited_out (1 would mean the wait completed), sets the device
 * error word, and returns; the next fa_check_device_status() then reports
 * FA_ERR_TIMEOUT and clears the word.  No trap, no hang, no fault. */
FA_API fa_status fa_selftest_wait_timeout(unsigned int limit_us, int* waited_out, fa_stream_t stream);

/* Self-test of the E4M3 quantiser's division (fa_quantize_fp8 divides every
 * element of a 64-row block by the block's scale s = amax / 448, [CH18]
 * §18.6.2): for n float32 device elements, q_fast[i] = x[i] / s[i % ns] by
 * the quantiser's shared-divisor method and q_ieee[i] = the IEEE float32
 * quotient; the two must agree bit for bit.  Device pointers; asynchronous on
 * `stream`. */
FA_API fa_status fa_selftest_quantiser_division(const float* x, const float* s, int ns, size_t n,
                                                float* q_fast, float* q_ieee, fa_stream_t stream);

/* ------------------------------------------------------ the plain calls */

/* bf16 forward ([FA2] §4 Algorithm 1).  q,k,v: bf16 inputs; o: bf16 output;
 * lse: float32 [B,H,N].  Tiles of 128 query rows x 128 keys (64 keys when
 * N <= 128). */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int N, int d, float scale, int causal,
                        const int* kv_lens, fa_stream_t stream);

/* Scratch for fa_bwd, in bytes: the row statistics LSE*log2(e) and
 * D = rowsum(dO*O) ([FA2] §5.2), 2 x [B,H,Np] float32, plus the float32 dQ
 * accumulator [B,H,Np,d] (Np = N rounded up to a multiple of 128).  0 for an
 * unsupported shape. */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/* bf16 backward of L = sum(O * dout) ([FA2] §5.4 Algorithm 2; [WIKI] §04):
 * given q, k, v, the forward's o and lse and the upstream gradient dout,
 * writes dq, dk, dv (bf16, overwritten, not accumulated).  Launches three
 * kernels on `stream`: preprocess (D and zeroed dQ accumulator), the main
 * kernel parallel over key blocks, and the dQ conversion. */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int B, int H, int N, int d, float scale, int causal, const int* kv_lens,
                        void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Number of 64-row scale blocks per (b,h): ceil(N / 64). */
FA_API int fa_fp8_num_blocks(int N);

/* Per-block E4M3 quantisation ([CH18] §18.6.2).  For each (b, h) and each
 * block of 64 consecutive rows x all d columns: amax = max|x|, s = amax / 448
 * (s = 1 when amax = 0), x8 = E4M3(x / s) with round-to-nearest-even and
 * saturation to +-448 (division and rounding in float32).
 *   x_bf16: bf16 [B,H,N,d]; x_e4m3: uint8 [B,H,N,d]; scales: float32
 *   [B,H,fa_fp8_num_blocks(N)]. */
FA_API fa_status fa_quantize_fp8(const void* x_bf16, void* x_e4m3, float* scales,
                                 int B, int H, int N, int d, fa_stream_t stream);

/* fa_quantize_fp8 of q [B,H,N,d], k and v [B,Hkv,N,d] in one launch (the
 * three inputs of the FP8 forward), same codes and scales as three separate
 * calls: sq [B,H,ceil(N/64)], sk, sv [B,Hkv,ceil(N/64)].
 * FA_ERR_INVALID_ARG if H % Hkv != 0. */
FA_API fa_status fa_quantize_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8,
                                     void* v8, float* sq, float* sk, float* sv, int B, int H, int Hkv,
                                     int N, int d, fa_stream_t stream);

/* FP8 forward: q8/k8/v8 are E4M3 [B,H,N,d] with per-64-row-block scales
 * sq/sk/sv (as written by fa_quantize_fp8), so that X ~= s_block * X8.
 * S = scale * (s_q s_k) (Q8 K8^T) accumulates in float32; the softmax runs in
 * float32; the probabilities are re-quantised to E4M3 (with the value scale of
 * each key block folded in) for the P V product; O is written as bf16 and LSE
 * as float32.  d must be 128. */
FA_API fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8,
                            const float* sq, const float* sk, const float* sv,
                            void* o, float* lse, int B, int H, int N, int d, float scale,
                            int causal, const int* kv_lens, fa_stream_t stream);

/* ------------------------------------------------ one call per pass */

/* Everything a forward or backward call needs.  Initialise with
 * fa_attn_params_init (which sets struct_size, the defaults below and zero
 * everywhere else), then fill in what the call uses.
 *
 *  struct_size   sizeof(fa_attn_params) as the caller compiled it; a
 *                mismatch (a caller built against another version of this
 *                header) is FA_ERR_INVALID_ARG.
 *  dtype         FA_BF16 (default); FA_F32: float32 tensors, [B,H,N,d] only,
 *                no mask beyond causal and kv_lens, computed through bf16
 *                tensor-core inputs (q and k split into bf16 high and low
 *                parts for the scores, x = hi + lo with ~16 significant bits;
 *                workspace from fa_attn_fwd_workspace_size); FA_E4M3:
 *                q, k, v E4M3 codes with q_scale, k_scale, v_scale
 *                [B, H or Hkv, ceil(N/64)], [B,H,N,d] with d = 128, no
 *                sliding window, block lists or N_q != N_k; o, dout bf16;
 *                the backward writes float32 dq, dk, dv and needs
 *                Hkv = H and deterministic = 0.
 *  layout        see fa_layout.
 *  batch         B, or the number of packed sequences.
 *  heads         H (query heads).
 *  kv_heads      Hkv key/value heads, H % Hkv == 0 (0 = H): grouped-query
 *                attention, multi-query for Hkv = 1 ([CH18] §18.7.1: K and V
 *                are broadcast over the heads; query head h uses key/value
 *                head h / (H / Hkv)); dk, dv hold the sum over the query
 *                heads sharing each key/value head.
 *  seqlen_q      N (N_q); packed: the longest query sequence (longer ones
 *                are cut to it).
 *  seqlen_k      N_k; 0 = the square kernels (N_k = N_q).  Nonzero with
 *                [B,H,N,d] selects rectangular attention (also when it equals
 *                N_q): decoding against a key/value cache (FlashDecoding,
 *                [CH18] §18.8.2) or cross-attention, the query rows of the
 *                heads sharing a key/value head processed as one block so
 *                that each K / V tile is read once per group; with causal the
 *                queries are the last N_q positions (query i sees keys
 *                j <= i + N_k - N_q).  Packed: the longest key range.
 *  head_dim      d: 64 or 128 (FA_E4M3: 128).
 *  total_q, total_k  packed tokens of q and of k (total_k 0 = total_q).
 *  scale         multiplies Q K^T (1/sqrt(d) for standard attention).
 *  causal        key j visible to query i only if j <= i (top-left aligned,
 *                N_q = N_k; see seqlen_k for N_q != N_k).
 *  window_left, window_right   sliding window (flash_attn_func's window_size,
 *                [CH18] §18.7.1): key j visible to query i only if
 *                i - window_left <= j <= i + window_right; -1 (default) =
 *                no bound on that side; below -1 is FA_ERR_INVALID_ARG.  Key
 *                blocks outside a tile's window are neither loaded nor
 *                multiplied ([CH18] §18.8.1).  Packed: within each sequence.
 *  kv_lens       [B] int32 valid keys per batch item (clamped to [0, N_k]),
 *                or NULL.  Not with the packed or [B,N,H,d] layouts.
 *  cu_seqlens_q, cu_seqlens_k   packed layout: device int32 [batch + 1],
 *                non-decreasing, starting at 0 (cu_seqlens_k NULL = the
 *                query ranges); with causal and separate key ranges the
 *                queries of a sequence are its last len_q positions.
 *  block_row_ptr, block_col_idx   block-sparse attention ([CH18] §18.8.1),
 *                [B,H,N,d] with N_q = N_k: query block i (128 rows) attends
 *                only to the 128-key blocks block_col_idx[block_row_ptr[i] ..
 *                block_row_ptr[i+1]-1] (ascending, no repeats, entries in
 *                [0, nb), nb = ceil(N/128)), on top of the causal and key
 *                padding masks; one list for every batch item and head; the
 *                kernels clamp the list bounds but do not otherwise validate
 *                the lists.  NULL = dense.
 *  num_splits    forward, [B,H,N,d] bf16 / E4M3 without Hkv != H, and the
 *                rectangular case: 0 = automatic split of the key sequence
 *                into ranges merged through the log-sum-exp ([CH18] §18.8.2;
 *                whole items first, only the remainder split, never for
 *                causal or key-padded square calls; rectangular calls with few
 *                items are split) -- the workspace must then hold
 *                fa_attn_fwd_workspace_size bytes; 1 (default) = no split;
 *                >= 2 = that many ranges per item (at most 64).
 *  block_c       forward, [B,H,N,d] bf16 / float32 without masks other than
 *                causal and kv_lens: keys per tile, 0 = automatic (128; 64
 *                when N <= 128), or 64 / 128.
 *  deterministic backward: bitwise-repeatable dq, dk, dv (flash_attn_func's
 *                `deterministic`, [CH18] §18.7.1): key block kt adds its dQ
 *                part to float32 accumulator kt % A (A = 1 .. 8, from the
 *                shape) on its turn, in increasing key-block order, and a last
 *                kernel sums the A accumulators in order.  Its CTAs wait on
 *                one another (bounded: FA_ERR_TIMEOUT through
 *                fa_check_device_status, never a hang), so two such calls must
 *                not overlap on one device.
 *  q, k, v, o, lse          forward inputs and outputs (backward: the
 *                forward's o and lse).
 *  q_scale, k_scale, v_scale   FA_E4M3 block scales.
 *  dout, dq, dk, dv         backward: upstream gradient and the gradients
 *                (overwritten, not accumulated).
 *  workspace, workspace_bytes   scratch of at least
 *                fa_attn_fwd_workspace_size / fa_attn_bwd_workspace_size
 *                bytes, 16-byte aligned (NULL allowed when that size is 0). */
typedef struct {
    size_t struct_size;
    fa_dtype dtype;
    fa_layout layout;
    int batch, heads, kv_heads, seqlen_q, seqlen_k, head_dim;
    int total_q, total_k;
    float scale;
    int causal;
    int window_left, window_right;
    int num_splits, block_c, deterministic;
    const int* kv_lens;
    const int* cu_seqlens_q;
    const int* cu_seqlens_k;
    const int* block_row_ptr;
    const int* block_col_idx;
    const void* q;
    const void* k;
    const void* v;
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    void* o;
    float* lse;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    void* workspace;
    size_t workspace_bytes;
} fa_attn_params;

/* Zero *p, then struct_size = sizeof(fa_attn_params), window_left =
 * window_right = -1, num_splits = 1. */
FA_API void fa_attn_params_init(fa_attn_params* p);

/* Workspace bytes fa_attn_fwd / fa_attn_bwd need for these parameters (the
 * tensor pointers are not read); 0 when none is needed or the combination is
 * refused (the call itself then reports why). */
FA_API size_t fa_attn_fwd_workspace_size(const fa_attn_params* p);
/* Key ranges per work item fa_attn_fwd will use for these parameters (1 = not
 * split; see num_splits).  The plan depends on the current device's SM count
 * (152 when no device is visible). */
FA_API int fa_attn_fwd_splits(const fa_attn_params* p);
FA_API size_t fa_attn_bwd_workspace_size(const fa_attn_params* p);

/* Forward pass ([FA2] §4 Algorithm 1) on the tensors and options in *p.
 * Combinations this library does not build (FA_ERR_UNSUPPORTED, refused
 * before any launch): FP8 with the packed or [B,N,H,d] layouts, a window,
 * block lists or N_q != N_k; float32 with any option beyond causal, kv_lens
 * and block_c; a window or block lists with N_q != N_k or with each other;
 * separate packed key ranges with a window; kv_lens with the packed or
 * [B,N,H,d] layouts; a split with shared key/value heads. */
FA_API fa_status fa_attn_fwd(const fa_attn_params* p, fa_stream_t stream);

/* Backward pass ([FA2] §5.4 Algorithm 2) of the forward with the same
 * parameters.  The same refusals as fa_attn_fwd, plus the FP8 backward with
 * shared key/value heads or deterministic.
 * FA_E4M3 ([CH18] §18.6.2): all five products of the backward run on FP8
 * tensor cores.  dout is quantised to E4M3 per 64-row block inside the call;
 * D = rowsum(dO^ * o) uses the dequantised dO^; P is rebuilt in float32 from
 * the E4M3 scores and re-quantised to E4M3 for dV = P^T dO^; dS = P * (dP - D)
 * is quantised to E5M2 with one power-of-two scale per (b, h), from a bound
 * on |dS|, for dK = dS^T Q^ and dQ = dS K^ (E5M2 x E4M3 products).  The block scales are
 * folded into the quantised operands; dq, dk, dv are float32 gradients with
 * respect to the dequantised inputs Q^ = s_q Q8, K^, V^. */
FA_API fa_status fa_attn_bwd(const fa_attn_params* p, fa_stream_t stream);

/* ---------------------------------------------- the backward's phases */

/* The three phases fa_bwd runs, callable one by one (bf16 tensors, same
 * workspace) so that each kernel can be timed on its own.
 * fa_bwd == fa_bwd_preprocess; fa_bwd_main; fa_bwd_dq.
 *   fa_bwd_preprocess: D = rowsum(dout * o) ([FA2] §5.2), LSE * log2(e) and
 *                      a zeroed float32 dQ accumulator, into `workspace`.
 *   fa_bwd_main:       the key-block-parallel kernel ([FA2] §5.4): writes
 *                      dk, dv and accumulates unscaled dQ into `workspace`.
 *   fa_bwd_dq:         dq = scale * accumulator, as bf16.
 * Each phase reads what the previous one wrote; call them in this order on
 * one stream (or order the streams). */
FA_API fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H, int N,
                                   int d, void* workspace, size_t workspace_bytes, fa_stream_t stream);
FA_API fa_status fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk,
                             void* dv, int B, int H, int N, int d, float scale, int causal,
                             const int* kv_lens, void* workspace, size_t workspace_bytes,
                             fa_stream_t stream);
FA_API fa_status fa_bwd_dq(void* dq, int B, int H, int N, int d, float scale, void* workspace,
                           size_t workspace_bytes, fa_stream_t stream);

/* Allocation-free backward (the pages have no counterpart: it only changes
 * where the scratch lives).  For callers that cannot allocate device memory,
 * e.g. a plugin inside a framework that owns the whole device-memory pool, or
 * a runtime that forbids allocation after start-up.  Same arguments and
 * results as fa_bwd, minus the workspace: the scratch is a fixed 128 MiB array
 * of device memory defined in this library, which every GPU that loads the
 * library keeps until the process exits.
 *   - Problems whose scratch (fa_bwd_workspace_size(...)) exceeds
 *     fa_bwd_noalloc_max_scratch() bytes are rejected with FA_ERR_INVALID_ARG.
 *   - The first call on each device looks up the array's device address (no
 *     allocation); make that first call before any stream capture.
 *   - Every call uses the same array and leaves its contents behind; each call
 *     re-initialises what it reads, but calls that overlap on the GPU (e.g. on
 *     two streams) race on it and must be serialised by the caller.
 *   - Calls no cudaMalloc / cudaFree and no allocating library routine. */
FA_API size_t fa_bwd_noalloc_max_scratch(void);
FA_API fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int H, int N, int d, float scale, int causal,
                                const int* kv_lens, fa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */

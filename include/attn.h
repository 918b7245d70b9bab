/*
 * attn.h -- C ABI of the GB300 (sm_103a) self-attention forward library.
 *
 * The operation.  For every batch b, query head a (key/value head g(a)) and
 * query position i:
 *
 *     s_ij  = scale * (q_i^(a) . k_j^(g(a)))          for every allowed key j
 *     O_i   = sum_j softmax_j(s_ij) * v_j^(g(a))
 *     LSE_i = ln sum_j exp(s_ij)                       (natural logarithm)
 *
 *   - Scaled dot-product attention Softmax(Q K^T / sqrt(d_k)) V and its
 *     row-wise softmax: "Trasformer 浅析" (atffang.github.io), section
 *     缩放点积注意力.  `scale` is applied exactly as passed; callers pass
 *     1/sqrt(d_k) for the textbook form.
 *   - Masks as an additive M with -inf entries (a -inf entry carries exactly
 *     zero weight): same page, section 填充掩码与因果掩码.  A disallowed pair is
 *     never evaluated; the mask is a predicate, not a stored matrix.
 *   - Shapes with H_q query heads sharing H_kv key/value heads through a map
 *     g(a): "Transformer 架构及其变体" (aaai.latere.ai), section
 *     带显式形状的因果自注意力.  This library fixes g(a) = a / (H_q / H_kv)
 *     (contiguous groups), the uniform grouping of "Transformer 演进与变体"
 *     (ai.icyfenix.cn), section GQA：分组查询注意力; H_kv = 1 is MQA and
 *     H_kv = H_q is MHA.
 *   - Sliding-window and local + global masks: "Transformer 演进与变体",
 *     section 稀疏注意力 (window of half-width w; global tokens attend to every
 *     position and every position attends to them).
 *
 * Tensor layouts (all contiguous, row-major, the head dimension fastest):
 *     Q, O : [B, H_q,  S, d_k]     K, V : [B, H_kv, S, d_k]     LSE : [B, H_q, S] float32
 * Element type: ATTN_BF16 -> Q, K, V, O are bfloat16 (fp32 accumulation);
 *               ATTN_F32  -> Q, K, V, O are float32;
 *               ATTN_FP8_E4M3 -> Q, K, V are E4M3 bytes, O is bfloat16.
 * Every pointer passed to attn_forward is a device pointer of the current
 * CUDA device and must be 16-byte aligned.
 *
 * Ownership: the caller owns Q, K, V, O, LSE and the stream.  A handle owns
 * its schedule, its tensor-map templates and, for the local + global mask, a
 * device scratch area sized at attn_create; attn_destroy frees them.
 *
 * Threading: a handle may be reused for any tensors of the shape it was
 * created for, on any stream, but not by two calls in flight at once (the
 * local + global scratch would be shared).  Distinct handles are independent.
 *
 * Errors: every entry point returns an attn_status.  Argument errors are
 * detected on the host before anything is launched.  attn_forward is
 * asynchronous: device-side watchdog errors (a bounded wait that ran out) are
 * recorded in the handle's device error word and read by
 * attn_poll_device_error, which synchronises the device.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,      /* a size, pointer, mask argument or scale is invalid  */
    ATTN_ERR_UNSUPPORTED = 2,      /* valid in principle but not built (e.g. d_k = 96)     */
    ATTN_ERR_CUDA = 3,             /* a CUDA runtime / driver call failed                  */
    ATTN_ERR_DEVICE_TIMEOUT = 4,   /* a kernel's bounded wait ran out (watchdog)           */
    ATTN_ERR_OOM = 5               /* device or host allocation failed at attn_create      */
} attn_status;

typedef enum {
    ATTN_MASK_FULL = 0,            /* every j                                              */
    ATTN_MASK_CAUSAL = 1,          /* j <= i                                               */
    ATTN_MASK_SLIDING = 2,         /* |i - j| <= window                                    */
    ATTN_MASK_CAUSAL_SLIDING = 3,  /* 0 <= i - j <= window  (window = max distance;       */
                                   /*  "4096 keys including self" is window = 4095)       */
    ATTN_MASK_LOCAL_GLOBAL = 4     /* |i - j| <= window, or i in G, or j in G              */
} attn_mask_kind;

/* ATTN_FP8_E4M3: Q, K, V are 8-bit E4M3 floats with per-tensor descale factors
 * (attn_set_fp8_descale); O is bfloat16.  The products run in E4M3 with fp32
 * accumulation, P is rounded to E4M3 for the second product, and the softmax is
 * fp32 ("Transformer 演进与变体" (ai.icyfenix.cn), section Flash Attention, FP8
 * support: matrix products in FP8, softmax and accumulation in higher precision;
 * "第 8 章 现代大模型架构", 8.6.5: scale before the multiply-add, descale at the
 * output).  Every mask kind, d_k = 64 or 128, with the ALiBi bias, a bias matrix
 * or neither. */
typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1, ATTN_FP8_E4M3 = 2 } attn_dtype;

typedef struct attn_plan* attn_handle;

/*
 * attn_create -- validate the problem, build the tile schedule on the host,
 * upload it, and allocate the handle's device buffers.
 *
 *   out        : receives the handle (set to NULL on failure).
 *   B, Hq, Hkv : batch, query heads, key/value heads; Hq % Hkv == 0.
 *   S          : sequence length, 1 <= S <= 1<<20.
 *   d_k        : head width; 64 or 128 (others: ATTN_ERR_UNSUPPORTED).
 *   dtype      : ATTN_BF16 or ATTN_F32.
 *   scale      : score multiplier, finite and > 0.
 *   kind       : mask kind.
 *   window     : half-width w (>= 0) for the window kinds, ignored otherwise.
 *   global_idx : host array of n_global positions in [0, S) (LOCAL_GLOBAL
 *                only; duplicates are removed; copied, the caller keeps it).
 *   n_global   : 0 <= n_global <= 4096; must be 0 for other kinds.
 * Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_OOM, ATTN_ERR_CUDA.
 */
attn_status attn_create(attn_handle* out, int B, int Hq, int Hkv, int S, int d_k,
                        attn_dtype dtype, float scale, attn_mask_kind kind, int window,
                        const int* global_idx, int n_global);

/*
 * attn_forward -- enqueue the forward pass on `stream` (a cudaStream_t, NULL
 * for the legacy default stream) and return without waiting.
 *
 *   Q, K, V : inputs in the layouts above.        O : output, same shape as Q.
 *   LSE     : float32 [B, Hq, S] output, or NULL to skip it.
 * Every row sees at least itself, so every O row is a convex combination of
 * V rows and every LSE entry is finite.
 * Errors: ATTN_ERR_INVALID_ARG (NULL handle or pointer, misaligned pointer),
 *         ATTN_ERR_CUDA (launch failure).  With the environment variable
 *         ATTN_DEBUG=1 the call synchronises and also reports
 *         ATTN_ERR_DEVICE_TIMEOUT.
 */
attn_status attn_forward(attn_handle h, const void* Q, const void* K, const void* V,
                         void* O, float* LSE, void* stream);

/* attn_destroy -- free the handle's device and host memory (synchronises the
 * device first).  NULL is accepted and ignored. */
attn_status attn_destroy(attn_handle h);

/* attn_status_string -- static English text of a status code. */
const char* attn_status_string(attn_status s);

/*
 * Schedule introspection (host only, no device work).
 *
 * The schedule is a list of work items of ATTN_WORK_INTS ints each:
 *   [0] bh          b * Hq + a  (query head a of batch b)
 *   [1] q_tile      query rows [q_tile * ATTN_TILE, (q_tile + 1) * ATTN_TILE) ∩ [0, S)
 *                   (for ATTN_WORK_GLOBAL_ROWS items: rows G[q_tile * ATTN_TILE + r])
 *   [2] kv_begin    first key tile evaluated (keys [kv * ATTN_TILE, ...))
 *   [3] kv_end      one past the last key tile evaluated
 *   [4] full_begin  key tiles in [full_begin, full_end) are FULL: every pair is
 *   [5] full_end    allowed and no mask is applied; the other tiles of
 *                   [kv_begin, kv_end) are PARTIAL and evaluate the mask predicate
 *   [6] flags       ATTN_WORK_GLOBAL_COLS: after the key tiles, also evaluate
 *                   the global keys G not inside the [kv_begin, kv_end) tiles,
 *                   gathered into narrow key tiles of at most ATTN_TILE keys;
 *                   ATTN_WORK_GLOBAL_ROWS: the item's rows are the global rows;
 *                   ATTN_WORK_HAS_GLOBAL_ROWS: the item's query tile holds rows of G,
 *                   whose outputs the item does not write
 *   [7] n_gtiles    number of gathered global-key tiles (ATTN_WORK_GLOBAL_COLS):
 *                   ceil(#(G outside the band) / ATTN_TILE);
 *                   for ATTN_WORK_GLOBAL_ROWS items: the index of the item's key
 *                   chunk.  The global rows' key tiles are split into chunks no
 *                   longer than the longest query-tile item (one item per chunk,
 *                   gathered row tile and head); each chunk yields a partial softmax
 *                   result and the chunk that finishes last combines them:
 *                   O = sum_c e^LSE_c O_c / sum_c e^LSE_c, LSE = ln sum_c e^LSE_c.
 * The query-tile items come first: the (batch, kv head) units in groups of
 * g = max(1, min(B*Hkv, 32 MiB / (512 S))) units (their K and V fit in 32 MiB at
 * d_k = 128), group after group, and within a group by decreasing number of tiles
 * (longest first), query heads of one kv head side by side.  When a group would
 * hold fewer than 4096 items (g * (Hq/Hkv) * ceil(S/ATTN_TILE)), all units form one
 * group.  For LOCAL_GLOBAL the
 * ATTN_WORK_GLOBAL_ROWS items follow them.  All items run in one launch: rows in G
 * are written only by ATTN_WORK_GLOBAL_ROWS items.
 */
#define ATTN_TILE 128
#define ATTN_WORK_INTS 8
#define ATTN_WORK_GLOBAL_COLS 1
#define ATTN_WORK_GLOBAL_ROWS 2
#define ATTN_WORK_HAS_GLOBAL_ROWS 4

/*
 * attn_schedule_host -- build the schedule attn_create would build for these
 * arguments, on the host only (no CUDA call; usable without a GPU).
 *   Arguments B .. n_global: as for attn_create (validated the same way).
 *   items   : output, room for `cap` items (cap * ATTN_WORK_INTS ints); may be
 *             NULL with cap = 0 to query the sizes only.
 *   n_items : receives the total number of items.
 *   n_first : receives the number of query-tile items; the remaining items are
 *             the ATTN_WORK_GLOBAL_ROWS chunks (all items run in one launch).
 * Returns ATTN_ERR_INVALID_ARG if cap is nonzero but smaller than the total.
 */
attn_status attn_schedule_host(int B, int Hq, int Hkv, int S, attn_mask_kind kind, int window,
                               const int* global_idx, int n_global, int* items, int cap,
                               int* n_items, int* n_first);

/*
 * attn_kv_schedule_host -- the key-tile schedule of the backward pass (host only).
 * One item of ATTN_WORK_INTS ints per key tile: [kv_tile, q_begin, q_end,
 * full_begin, full_end, 0, 0, 0]: the query tiles [q_begin, q_end) hold every row
 * that may see a key of the tile, and in [full_begin, full_end) every (row, key)
 * pair is allowed.  Longest first.  items may be NULL with cap = 0 to query the count.
 * Errors: ATTN_ERR_INVALID_ARG; ATTN_ERR_UNSUPPORTED for LOCAL_GLOBAL.
 */
attn_status attn_kv_schedule_host(int S, attn_mask_kind kind, int window, int* items, int cap, int* n_items);

/*
 * attn_bwd_dq_schedule_host -- the work items of the backward's dQ launch (host only):
 * the first-launch items of attn_schedule_host for these arguments (no global tokens),
 * stably regrouped so that the items of the kv heads whose K and V fit in 32 MB
 * (kv_group = max(1, 32 MiB / (4 S d_k)) heads) run together, group by group in
 * (batch, kv head) order; within a group the forward's longest-first order is kept.
 * items may be NULL with cap = 0 to query the count.
 * Errors: ATTN_ERR_INVALID_ARG (bad shape, LOCAL_GLOBAL, cap too small).
 */
attn_status attn_bwd_dq_schedule_host(int B, int Hq, int Hkv, int S, int d_k, attn_mask_kind kind, int window,
                                      int* items, int cap, int* n_items);

/*
 * attn_bwd_lg_lists_host -- the per-tile lists both backward kernels walk under
 * ATTN_MASK_LOCAL_GLOBAL (host only).  The mask |i - j| <= window, or i in G, or j in G
 * ("Transformer 演进与变体" (ai.icyfenix.cn), section 稀疏注意力: global tokens attend
 * to and are attended by every position) is symmetric, so one list per tile index x
 * (0 <= x < n_tiles = ceil(S / ATTN_TILE)) gives both the key tiles of query tile x (dQ)
 * and the query tiles of key tile x (dK, dV): ascending, every tile t holding at least
 * one allowed pair against x, each entry t | ATTN_LIST_FULL when every pair of the two
 * tiles lies inside [0, S) and is allowed.
 *   globals  : global positions (any order, duplicates allowed), each in [0, S).
 *   list     : output, room for `cap` entries; may be NULL with cap = 0 to query n_list.
 *   offsets  : output, n_tiles + 1 ints (entries of tile x: offsets[x] .. offsets[x+1]-1);
 *              may be NULL when cap = 0.
 * Errors: ATTN_ERR_INVALID_ARG (bad S, window or position; cap nonzero but too small).
 */
#define ATTN_LIST_FULL (1 << 16)
attn_status attn_bwd_lg_lists_host(int S, int window, const int* globals, int n_global, int* list, int cap,
                                   int* offsets, int* n_list);

/*
 * attn_poll_device_error -- synchronise the device, read the handle's device
 * error word into *code (0 = none, otherwise a bit set of the role whose
 * bounded wait ran out), clear it, and return ATTN_ERR_DEVICE_TIMEOUT if it
 * was nonzero.
 */
attn_status attn_poll_device_error(attn_handle h, int* code);

/*
 * attn_selftest_exp2 -- test hook: y[i] = the exp2 approximation the library's
 * FMA-pipe exponential evaluates (range reduction x = j + f, j = round(x), and a
 * degree-3 polynomial for 2^f on [-1/2, 1/2], max relative error 7.5e-5 for
 * x >= -125; inputs below -125 are clamped to -125).  x, y: device float
 * arrays of n elements; enqueued on `stream`.  Errors: ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_CUDA.
 */
attn_status attn_selftest_exp2(const float* x, float* y, int n, void* stream);

/*
 * attn_selftest_device_once -- host-only test hook of the per-device set-up registry
 * the launchers use for kernel attributes (the dynamic shared-memory opt-in belongs to
 * a device context, so it is made once per device and kernel, not once per process).
 * Exercises the registry with fake device ids from several host threads: each
 * (device, kernel, value) entry must run its set-up exactly once, a failed set-up must
 * run again on the next call, and distinct devices must not share entries.  Touches no
 * GPU.  Returns 0 when every check holds, else the number of the first failed check.
 */
int attn_selftest_device_once(void);

/*
 * attn_set_alibi -- add the ALiBi score bias to every later attn_forward of this
 * handle: logits_ij = scale * q_i . k_j + b_ij with b_ij = -slopes[a] * |i - j|.
 *   - The additive-bias form logits = q.k / sqrt(d_k) + b_ij and ALiBi's
 *     -m_h (i - j), j <= i: "Transformer 架构及其变体" (aaai.latere.ai), sections
 *     加性偏置：ALiBi and the unified view of sequence and graph attention; the
 *     distance form -m |i - j|: "Trasformer 浅析" (atffang.github.io), section
 *     线性偏置注意力.  The pages fix one slope per head but give no values.
 *   slopes : HOST array of Hq finite floats (query head a uses slopes[a]; copied),
 *            or NULL to remove the bias.
 * The bias enters the row max, the weights and the LSE (LSE = ln sum_j e^{logits_ij}).
 * Every mask kind and every dtype takes it; under LOCAL_GLOBAL the global keys and rows
 * get the same distance term (|i - j| between the positions of the pair); with E4M3
 * inputs it joins the descaled scores, element by element.
 * Errors: ATTN_ERR_INVALID_ARG (NULL handle, non-finite slope),
 *         ATTN_ERR_UNSUPPORTED (a bias matrix set), ATTN_ERR_OOM, ATTN_ERR_CUDA.
 * Must not be called while a forward of this handle is in flight.
 */
attn_status attn_set_alibi(attn_handle h, const float* slopes);

/*
 * attn_set_bias -- add a given bias matrix to the scores of every later attn_forward of
 * this handle: logits_ij = scale * q_i . k_j + b_ij with b_ij = bias[b', a', i, j], the
 * general b_ij of the unified biased-logits form ("Transformer 架构及其变体"
 * (aaai.latere.ai), the unified view of sequence and graph attention: the scaled
 * scores plus a bias b_ij, of which ALiBi's distance penalty is one instance).
 *   bias : DEVICE bf16 tensor [Bb, Hb, S, ld], 16-byte aligned, owned by the caller and
 *          read by every later forward (it must stay valid and unchanged while they run);
 *          NULL removes the bias.
 *   Bb   : 1 (one matrix for every batch entry) or B;  b' = (Bb == 1 ? 0 : b).
 *   Hb   : 1 (one matrix for every query head) or Hq;  a' = (Hb == 1 ? 0 : a).
 *   ld   : row stride in elements, >= S and a multiple of 8 (rows may be padded; the
 *          padding is never used for the result).
 * Masked pairs stay masked whatever their bias; the bias enters the row max, the
 * weights and the LSE.  Every mask kind takes it; under LOCAL_GLOBAL the global keys and
 * the global rows read b_ij at their own positions.
 * With ATTN_FP8_E4M3 inputs the bias is added to the descaled scores, in the same
 * logit units.
 * Errors: ATTN_ERR_INVALID_ARG (NULL handle, misaligned pointer, Bb / Hb / ld out of
 *         range); ATTN_ERR_UNSUPPORTED (ATTN_F32 inputs, or with the ALiBi bias set).
 * attn_backward of a handle with a bias matrix recomputes P with the same b_ij.
 * Must not be called while a forward of this handle is in flight.
 */
attn_status attn_set_bias(attn_handle h, const void* bias, int Bb, int Hb, long ld);

/*
 * attn_backward -- the gradients of the forward pass of this handle with respect to
 * Q, K and V, for the output gradient dO:
 *     P_ij = exp(s_ij - LSE_i), D_i = dO_i . O_i, dS_ij = P_ij (dO_i . v_j - D_i),
 *     dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i,
 * with dK and dV summed over the query heads of each kv head (g(a) as in the forward).
 * The pages give no backward formulas; they describe the tiled forward as exact and used
 * to train models ("Transformer 演进与变体" (ai.icyfenix.cn), section Flash Attention),
 * so this is the derivative of the definition.  P is recomputed tile by tile from the
 * saved LSE; nothing of size S x S is stored.
 *   Q, K, V, O, dO : bf16 device tensors in the forward layouts; O and LSE are the
 *                    outputs of attn_forward for these Q, K, V.
 *   LSE            : float32 [B, Hq, S] device array (required).
 *   dQ, dK, dV     : bf16 outputs with the shapes of Q, K, V (overwritten).
 * With the ALiBi bias set (attn_set_alibi), s_ij includes -m_a |i - j| as in the forward,
 * and with a bias matrix set (attn_set_bias) it includes b_ij, read from the caller's
 * bias tensor, which must still hold the values the forward used (neither bias depends
 * on Q or K, so each enters only the recomputed P).
 * Enqueued on `stream`; the first call allocates the handle's backward scratch
 * (2 * B*Hq*ceil(S/128)*128 floats and the key-tile schedule).
 * Under ATTN_MASK_LOCAL_GLOBAL both kernels walk per-tile lists of partner tiles
 * (attn_bwd_lg_lists_host) with the window plus the global rows and columns as a bit
 * mask; a global row's dQ and a global key's dK, dV take every position.
 * Errors: ATTN_ERR_INVALID_ARG (NULL or misaligned pointer); ATTN_ERR_UNSUPPORTED
 * (dtype other than ATTN_BF16); ATTN_ERR_OOM; ATTN_ERR_CUDA.
 */
attn_status attn_backward(attn_handle h, const void* Q, const void* K, const void* V, const void* O,
                          const float* LSE, const void* dO, void* dQ, void* dK, void* dV, void* stream);

/*
 * attn_set_fp8_descale -- the per-tensor factors of an ATTN_FP8_E4M3 handle: the
 * real Q is descale_q times the stored E4M3 values, and likewise K and V.  Scores
 * are scale * descale_q * descale_k * (q8 . k8); O = descale_v * sum_j p_j v8_j / l.
 * Defaults 1.  Errors: ATTN_ERR_INVALID_ARG (not an E4M3 handle; a factor that is
 * not finite and > 0).  Must not be called while a forward of the handle is in flight.
 */
attn_status attn_set_fp8_descale(attn_handle h, float descale_q, float descale_k, float descale_v);

/*
 * attn_set_watchdog -- test hook for the failure-detection path.
 *   limit_ns : wall-clock limit of every bounded wait inside the kernels
 *              (default 2e9 ns).
 *   withhold : 0 = normal; 1 = the producer of the tensor-core kernel never
 *              loads V, so the first wait for V runs out: the kernel records
 *              ATTN_ERR_DEVICE_TIMEOUT in the error word, releases its tensor
 *              memory and returns (output contents are then undefined).
 */
attn_status attn_set_watchdog(attn_handle h, long long limit_ns, int withhold);

/*
 * attn_forward_noalloc -- the bf16 forward pass for callers that cannot
 * allocate device memory (no cudaMalloc, no cudaFree, no allocating library
 * call): code running inside a memory pool it does not own, runtimes that
 * forbid allocation after start-up, processes whose device footprint must stay
 * fixed.  The pages describe no such interface; it is a deployment
 * convenience of this library.
 *
 *   B .. n_global : as for attn_create with dtype ATTN_BF16 (validated the same
 *                   way; the schedule is built on the host on every call).
 *   Q, K, V, O, LSE, stream : as for attn_forward (caller-owned device
 *                   buffers; LSE may be NULL).
 *
 * Instead of handle-owned buffers, the call keeps its scratch (error word,
 * work list, global-token list and bits, and for the local + global mask the
 * partial results and arrival counters of the global-row chunks) in one fixed
 * device array of ATTN_NOALLOC_SCRATCH_BYTES, a file-scope __device__ object
 * that every GPU which loads this library holds until the process exits.
 * A problem whose scratch does not fit returns ATTN_ERR_UNSUPPORTED before
 * anything is launched (the work list takes 32 bytes per (batch, head,
 * 128-row tile); the local + global mask adds B*Hq*n_global*chunks*(d_k+1)*4
 * bytes of partial results of the chunked global rows).
 *
 * The first call on a device looks up the array's address (once per device,
 * with that device current); make that first call before any stream capture.
 * Every call shares the one array and leaves its contents behind: calls that
 * overlap on the GPU (two streams, or two host threads) race and must be
 * serialised by the caller.  The call passes its schedule to the device inside
 * kernel parameters (copied by the launch; no host buffer is read after the
 * call returns), clears the counters that must start at zero, and returns
 * without waiting for the kernels.  Device watchdog bits of every call collect
 * in the array's error word until attn_forward_noalloc_poll_error reads them.
 * Errors: as attn_create and attn_forward, plus ATTN_ERR_UNSUPPORTED above.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
attn_status attn_forward_noalloc(int B, int Hq, int Hkv, int S, int d_k, float scale,
                                 attn_mask_kind kind, int window, const int* global_idx,
                                 int n_global, const void* Q, const void* K, const void* V,
                                 void* O, float* LSE, void* stream);

/*
 * attn_forward_noalloc_poll_error -- synchronise the device, read the error word
 * of attn_forward_noalloc's scratch array on the current device into *code
 * (0 = none, otherwise a bit set of the kernel roles whose bounded wait ran
 * out, collected over every call since the last poll), clear it, and return
 * ATTN_ERR_DEVICE_TIMEOUT if it was nonzero.  Allocates nothing.  The outputs of
 * a call that set a bit are undefined.  Errors: ATTN_ERR_INVALID_ARG (code NULL),
 * ATTN_ERR_CUDA.
 */
attn_status attn_forward_noalloc_poll_error(int* code);

/*
 * attn_forward_noalloc_set_watchdog -- test hook of attn_forward_noalloc, as
 * attn_set_watchdog for a handle: limit_ns bounds every wait inside its kernels
 * (default 2e9 ns), withhold = 1 makes the producer never load V so the first
 * wait for V runs out.  Applies to the calls made after it, process-wide.
 * Errors: ATTN_ERR_INVALID_ARG (limit_ns <= 0, withhold not 0 or 1).
 */
attn_status attn_forward_noalloc_set_watchdog(long long limit_ns, int withhold);

/*
 * ---------------------------------------------------------------- decode
 * Decode / key-value-cache attention: S_q new query rows per sequence
 * against a cache of keys and values.
 *
 *   - The step-t output Softmax(q_t K_{1:t}^T / sqrt(d_k)) V_{1:t} of a new
 *     query against every cached key and value: "Trasformer 浅析"
 *     (atffang.github.io), section 推理：KV 缓存.
 *   - Ragged batches (sequence r holds S_r cached positions) and prefill run in
 *     chunks: "第 8 章 现代大模型架构" (theaiera.top), section
 *     预填充创建缓存，解码复用缓存.  Row i of sequence b is the position
 *     t = cache_len[b] - S_q + i; its own key and value are already in the cache.
 *   - Cross-attention (queries from the decoder, keys and values from the
 *     encoder, an n_dec x n_enc score matrix): "Trasformer 浅析", section
 *     交叉注意力.  Use ATTN_MASK_FULL with the encoder output as the cache.
 *
 * Mask kinds: ATTN_MASK_FULL (every j < cache_len[b]), ATTN_MASK_CAUSAL
 * (j <= t), ATTN_MASK_CAUSAL_SLIDING (t - window <= j <= t).  The other kinds
 * return ATTN_ERR_UNSUPPORTED.
 *
 * Layouts (contiguous, head dimension fastest, bfloat16):
 *     Q, O : [B, Hq, S_q, d_k]     K, V (the cache) : [B, Hkv, S_cap, d_k]
 *     LSE  : [B, Hq, S_q] float32 (natural logarithm), may be NULL.
 * Cache positions at or past cache_len[b] are never used; they may hold
 * anything, NaN included.
 *
 * Limits: B <= ATTN_DECODE_MAX_BATCH; (Hq / Hkv) * S_q <= ATTN_DECODE_MAX_ROWS
 * (all query rows of a kv head's group go through one tile); d_k 64 or 128.
 *
 * Ownership and threading as for attn_create: the handle owns an error word,
 * the arrival counters and the partial-result area of split sequences; a
 * handle must not be used by two calls in flight at once.
 */
#define ATTN_DECODE_MAX_BATCH 1024
#define ATTN_DECODE_MAX_ROWS 64
typedef struct attn_decode_plan* attn_decode_handle;

/*
 * attn_decode_create -- validate the shape and allocate the handle.
 *   B, Hq, Hkv : batch (1 .. ATTN_DECODE_MAX_BATCH), query heads, kv heads
 *                (Hq % Hkv == 0; query head a uses kv head a / (Hq / Hkv)).
 *   S_q        : new query rows per sequence (>= 1).
 *   S_cap      : cache capacity in positions (>= 1; >= S_q for the causal kinds).
 *   d_k, scale, kind, window : as for attn_create (window: CAUSAL_SLIDING only).
 * Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_OOM, ATTN_ERR_CUDA.
 */
attn_status attn_decode_create(attn_decode_handle* out, int B, int Hq, int Hkv, int S_q, int S_cap,
                               int d_k, float scale, attn_mask_kind kind, int window);

/*
 * attn_decode_forward -- enqueue one decode step on `stream` and return.
 *   Q, K, V, O, LSE : device pointers (16-byte aligned) in the layouts above.
 *   cache_len       : HOST array of B lengths, each in [1, S_cap], and >= S_q
 *                     for the causal kinds; read before the call returns.
 * The (sequence, kv head) units are laid end to end as one list of 128-key
 * tiles and a persistent grid (one CTA per multiprocessor; two at d_k = 64
 * with at most 32 packed rows) takes contiguous shares of it, weighted by tiles and by the units begun inside a share
 * (attn_decode_schedule_host); a unit cut between CTAs is combined on the
 * device by a second, small kernel enqueued behind the first (see
 * attn_decode_set_merge_mode).
 * Errors: ATTN_ERR_INVALID_ARG (pointers, lengths), ATTN_ERR_CUDA.  Device
 * watchdog errors are read by attn_decode_poll_device_error; the outputs of
 * that call are then undefined (the poll resets the handle's counters, so the
 * handle stays usable).
 */
attn_status attn_decode_forward(attn_decode_handle h, const void* Q, const void* K, const void* V,
                                const int* cache_len, void* O, float* LSE, void* stream);

/* attn_decode_poll_device_error -- as attn_poll_device_error, for a decode handle. */
attn_status attn_decode_poll_device_error(attn_decode_handle h, int* code);

/*
 * attn_decode_set_alibi -- as attn_set_alibi, for a decode handle: the bias of a
 * query row at position t is -slopes[a] * |t - j| (t = cache_len[b] - S_q + i).
 * NULL removes it.  Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_OOM, ATTN_ERR_CUDA.
 */
attn_status attn_decode_set_alibi(attn_decode_handle h, const float* slopes);

/*
 * attn_decode_set_grid_limit -- test hook: run at most max_ctas CTAs (>= 1) per
 * launch instead of one per multiprocessor, so that small problems exercise long
 * shares spanning several units.  Errors: ATTN_ERR_INVALID_ARG.
 */
attn_status attn_decode_set_grid_limit(attn_decode_handle h, int max_ctas);

/*
 * attn_decode_set_merge_mode -- where the partial results of a unit (b, g) split over
 * several CTAs are combined (O = sum_c e^{LSE_c - M} O_c / W, LSE = M + ln W with
 * M = max_c LSE_c, W = sum_c e^{LSE_c - M}, the same merge either way):
 *   0 (default): by a second, small kernel (one warp per packed row), launched as a
 *                programmatic dependent of the decode kernel so that its launch overlaps
 *                the decode kernel; it is not enqueued when no unit is split;
 *   1          : by the last CTA to finish a part of the unit, inside the decode kernel;
 *   2          : by the merge kernel (as 0).
 * Errors: ATTN_ERR_INVALID_ARG (NULL handle, mode outside 0..2).
 */
attn_status attn_decode_set_merge_mode(attn_decode_handle h, int mode);

/*
 * attn_decode_launch_count -- *n = the number of kernels the last attn_decode_forward of
 * this handle enqueued (1, or 2 with the merge kernel; 0 before the first call).
 * Errors: ATTN_ERR_INVALID_ARG (NULL argument).
 */
attn_status attn_decode_launch_count(attn_decode_handle h, int* n);

/* attn_decode_destroy -- free the handle (synchronises the device first); NULL is ignored. */
attn_status attn_decode_destroy(attn_decode_handle h);

/*
 * attn_decode_schedule_host -- the work split attn_decode_forward uses, on the
 * host only (no CUDA call).  Sequence b needs the key tiles [lo_b, hi_b) with
 * hi_b = ceil(cache_len[b] / ATTN_TILE) and lo_b = 0, or for CAUSAL_SLIDING
 * lo_b = max(0, cache_len[b] - S_q - window) / ATTN_TILE.  With
 * n_b = hi_b - lo_b, tile_prefix[b] = n_0 + ... + n_{b-1}; unit (b, g) covers
 * the indices [Hkv * tile_prefix[b] + g * n_b, ... + n_b) of one list of
 * T = Hkv * tile_prefix[B] tiles.  CTA k of the *n_cta = min(n_sm, 512, T) CTAs
 * takes the indices [share[k], share[k + 1]): share[0] = 0, share[n_cta] = T,
 * every share non-empty, and the boundaries sit at equal steps of
 * F(i) = i + 2 * (number of unit begins u with 0 < u <= i), so that a share's
 * weight is its tiles plus two for every unit it begins inside it (the cost of
 * one more stretch: an epilogue and a pipeline refill, about two tiles' time).
 *   tile_prefix : output, B + 1 ints.
 *   share       : output, *n_cta + 1 long longs (room for min(n_sm, 512) + 1).
 * n_sm is the CTA budget: attn_decode_forward passes the multiprocessor count,
 * or twice it at d_k = 64 with at most 32 packed rows.
 * Errors: ATTN_ERR_INVALID_ARG (n_sm < 1, NULL outputs, shape or lengths as for
 * the calls above).
 */
attn_status attn_decode_schedule_host(int B, int Hkv, int S_q, int S_cap, attn_mask_kind kind, int window,
                                      const int* cache_len, int n_sm, int* n_cta, int* tile_prefix,
                                      long long* share);

#ifdef __cplusplus
}
#endif
#endif /* GB300_ATTN_H */

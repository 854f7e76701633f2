/*
 * fa_prefill.h -- C ABI of the GB300 (sm_103a) causal prefill flash-attention
 * library, libfa_prefill.so.
 *
 * The operation is the prefill attention forward pass of a llama-style
 * inference engine:
 *
 *     O = softmax(scale * Q K^T + causal mask) V
 *
 * over 16-bit Q, K, V with f32 accumulation, computed tile by tile with an
 * online softmax (running row max m and row sum l, O rescaled when m moves).
 * The pages this follows describe that kernel as one launcher call per layer
 * returning an int status (minfer "49 · r46 (FAP1) — FA audit +
 * occupancy/bank-conflict levers", section 3.2, the launcher), the validity
 * mask "key column at or before the query position AND inside the stored KV
 * range" (minfer "28 · r23 — f16-path whole-graph wall decomposition + FA_TKV
 * occupancy raise", section 3.2), the KV-head index passed per query head and
 * the online softmax with its -inf guard (minfer "53 · r50 — FA_TKV 32->16
 * occupancy experiment", sections 2 and 3.2), and the rule that resource
 * limits must fail loudly rather than fall back silently (minfer "11 · P5 —
 * prefill gap session: TM=128 big tiles + FA rewrite", section 3.3).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout ("BSHD", contiguous, hd fastest):
 *     q, o : [B][Sq][Hq][hd]        k, v : [B][Skv][Hkv][hd]
 * GQA: query head hq reads KV head hq / (Hq / Hkv); Hq must be a multiple of Hkv.
 * Causal alignment is bottom-right: the Sq query rows are the LAST Sq positions
 * of the Skv keys, so query row i sees key j iff j <= (Skv - Sq) + i.  With
 * Sq == Skv this is the usual lower-triangular mask; with Sq < Skv it is a
 * chunk of new rows attending to a cached prefix plus themselves.  A row that
 * sees no key (possible only when causal and Skv < Sq) gets O = 0.
 * causal == 0 makes every row see all Skv keys.
 * scale multiplies Q K^T before the mask and the softmax; it must be finite and
 * > 0 (1/sqrt(hd) is the usual value).
 *
 * Supported: hd any multiple of 8 from 8 to 256 (16-byte rows for TMA).  A
 * head runs on the kernel of the next width up, 64, 128 or 256 columns: its
 * tensor maps describe the true width, so TMA loads the missing columns of Q,
 * K and V as zeros and clips them from O, which leaves S and P V unchanged
 * (the tensor work is that of the wider kernel).  Heads over 128 wide run on
 * the one-shot kernel only (fa_prefill, fa_prefill_bf16, fa_prefill_ex and
 * fa_prefill_kvcache without a workspace); the split-KV, paged and
 * static-scratch entry points take heads up to 128 wide.  Any B, Sq, Skv >= 0 and
 * Hq, Hkv >= 1 whose tensors fit TMA's 32-bit coordinates.  B == 0 or Sq == 0
 * is a no-op
 * returning FA_OK (the pointers may then be NULL: nothing is read or written);
 * Skv == 0 writes O = 0 (k and v may then be NULL).
 *
 * Memory and ownership: q, k, v, o are DEVICE pointers owned by the caller,
 * 16-byte aligned, on the current CUDA device; o must not overlap q, k or v.
 * The library allocates no device memory, keeps no per-call state and never
 * frees caller memory.  It caches, per device, the kernel attributes it has
 * set and the driver entry point it uses to encode TMA descriptors.
 *
 * Asynchrony: each call validates its arguments on the host, encodes the TMA
 * descriptors, and enqueues ONE kernel on `stream` (a cudaStream_t; NULL means
 * the legacy default stream).  It returns once the launch is enqueued; the
 * result is ready when the stream reaches that point.  Errors that happen while
 * the kernel runs surface at the caller's next synchronisation; a pipeline
 * watchdog inside the kernel (see fa_debug_status) turns a stalled wait into a
 * recorded status instead of a hang.
 *
 * Errors are returned, never printed and ignored: every entry point returns
 * FA_OK (0) or one of the fa_status_t codes below, and on any error no kernel
 * was launched.
 *
 * Entry points
 * ------------
 *   fa_prefill, fa_prefill_bf16      one-shot kernel (hd 8 .. 256, multiples of 8)
 *   fa_prefill_ws, fa_prefill_ws_bf16  split-KV kernel with a caller workspace
 *   fa_workspace_bytes               its workspace size
 *   fa_split_kv_advised(_hd)         whether to take split-KV for a shape
 *   fa_prefill_ex                    either kernel, any hd, optional log-sum-exp
 *   fa_prefill_kvcache               attention over a K/V cache of capacity kv_cap
 *   fa_prefill_paged, fa_prefill_paged_ws  attention over a paged K/V pool
 *   fa_kv_append                     write new tokens' K/V rows into a cache
 *   fa_prefill_ws_static             split-KV with library-owned scratch
 *   fa_status_string, fa_smem_bytes, fa_debug_status(_clear)  diagnostics
 *   fa_debug_set_watchdog_ns         testing hook: the kernels' wait limit
 *   fa_debug_force_path              testing hook: which kernel runs
 *   fa_debug_schedule                the split-KV work split for a shape
 *   fa_debug_row_pairing             the one-shot grid's pairing of query tiles
 */
#ifndef FA_PREFILL_H
#define FA_PREFILL_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer (where one is read or written),
                                negative size, Hq or Hkv < 1,
                                Hq % Hkv != 0, non-finite or <= 0 scale,
                                o overlapping q/k/v                        */
    FA_ERR_UNSUPPORTED = 2,  /* hd not supported by the entry point, or a tensor too large
                                for TMA's 32-bit coordinates               */
    FA_ERR_ALIGNMENT = 3,    /* a pointer not 16-byte aligned (TMA rule)  */
    FA_ERR_SMEM = 4,         /* the kernel's shared-memory request does not
                                fit the device, or setting it failed        */
    FA_ERR_LAUNCH = 5,       /* the launch (or TMA descriptor encode) failed */
    FA_ERR_DEVICE = 6,       /* no current device, or not an sm_103 GPU    */
    FA_ERR_SCRATCH = 7       /* fa_prefill_ws_static only: the call needs
                                more than FA_STATIC_SCRATCH_BYTES of scratch */
} fa_status_t;

/*
 * fa_prefill -- f16 Q/K/V/O (IEEE binary16), f32 accumulation.
 *   q      [B][Sq][Hq][hd]  f16, device, read-only
 *   k, v   [B][Skv][Hkv][hd] f16, device, read-only
 *   o      [B][Sq][Hq][hd]  f16, device, written (every element)
 *   causal 0 or 1 (any non-zero value means 1)
 *   scale  softmax scale applied to Q K^T
 *   stream cudaStream_t to enqueue on (NULL = legacy default stream)
 * Returns FA_OK or an fa_status_t error (nothing launched on error).
 */
int fa_prefill(const void* q, const void* k, const void* v, void* o,
               int B, int Hq, int Hkv, int Sq, int Skv, int hd,
               int causal, float scale, void* stream);

/* fa_prefill_bf16 -- identical to fa_prefill with bfloat16 Q/K/V/O. */
int fa_prefill_bf16(const void* q, const void* k, const void* v, void* o,
                    int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                    int causal, float scale, void* stream);

/*
 * fa_prefill_ws / fa_prefill_ws_bf16 -- the same operation computed by a
 * load-balanced split-KV schedule: at most one CTA per SM.  With no more
 * query-tile pairs than SMs, each pair is cut into near-equal pieces of its
 * KV steps and every CTA computes one piece (the split-KV kernel); with more
 * pairs, the CTAs are persistent and each takes an equal contiguous share of
 * all (query-tile pair, KV tile) steps ("stream-K", the persistent kernel,
 * whose epilogue warpgroup writes one segment's output while the next
 * segment's steps run).  Either way short prompts, single heads, causal rows
 * of very different lengths and grids of a few more pairs than SMs keep
 * every SM busy.  A
 * query-tile pair whose KV steps are split between CTAs is merged
 * by a second, short kernel enqueued behind the first (programmatic dependent
 * launch), over the whole GPU and in a fixed order (results are
 * deterministic, run to run); this is the
 * split-K with a fixed-order reduction and no atomic accumulation that the
 * pages' GEMM work uses for underfilled grids, applied to the KV dimension.
 * The merge keeps each piece's unnormalised O with its running max m and sum
 * l, the state of the online softmax (minfer "53 · r50 — FA_TKV 32->16
 * occupancy experiment", section 2), and combines pieces exactly as the
 * online softmax combines tiles.
 *
 * The first 13 arguments are those of fa_prefill / fa_prefill_bf16, then:
 *   workspace        caller-owned DEVICE memory, >= fa_workspace_bytes(hd)
 *                    bytes, 256-byte aligned; no initialisation needed (a
 *                    call reads only what it wrote itself)
 *   workspace_bytes  its size in bytes
 * Calls that share one workspace must not overlap on the GPU (issue them on
 * one stream, or give each stream its own workspace).  No CTA waits on
 * another: the pieces meet only in the merge kernel.
 * Additional errors: FA_ERR_INVALID_ARG for a NULL or too small workspace,
 * FA_ERR_ALIGNMENT for a workspace not 256-byte aligned.
 */
int fa_prefill_ws(const void* q, const void* k, const void* v, void* o,
                  int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                  int causal, float scale, void* workspace,
                  size_t workspace_bytes, void* stream);

int fa_prefill_ws_bf16(const void* q, const void* k, const void* v, void* o,
                       int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                       int causal, float scale, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Workspace bytes fa_prefill_ws needs for head dimension hd (0 if
 * unsupported, or over 128); those of the 64- or 128-column kernel the head
 * runs on, independent of the other sizes: 512 piece slots (a CTA of at
 * most 256 holds at most two pieces of split pairs), each with both query
 * tiles' partial O (f32, 128 rows x kernel width) and m and l per row, i.e.
 * 512 * (1024 * width + 2048) bytes.  Host-only. */
size_t fa_workspace_bytes(int hd);

/*
 * fa_prefill_ex -- one entry point for every head dimension and both kernels,
 * with an optional per-row log-sum-exp output:
 *   q, k, v, o, B ... scale   as fa_prefill
 *   lse        NULL, or DEVICE float [B][Hq][Sq], 4-byte aligned, written:
 *              lse[b][hq][i] = log sum_j exp(scale * q_i . k_j) over the keys
 *              row i sees (-inf for a row that sees none) -- the online
 *              softmax's running max and sum taken together (minfer "53 · r50
 *              — FA_TKV 32->16 occupancy experiment", section 2), which is
 *              what combines attention computed over separate key ranges
 *   bf16       0: f16, non-zero: bfloat16
 *   workspace  NULL: the one-shot kernel (any supported hd); otherwise the
 *              split-KV kernel under fa_prefill_ws's rules (hd up to 128)
 * Errors: those of fa_prefill / fa_prefill_ws, FA_ERR_ALIGNMENT for a
 * misaligned lse, FA_ERR_INVALID_ARG for lse overlapping q, k, v, o or the
 * workspace.
 */
int fa_prefill_ex(const void* q, const void* k, const void* v, void* o,
                  float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                  int causal, float scale, int bf16, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * fa_split_kv_advised -- host-only advice on which kernel to call for a shape
 * on the current device: 1 if fa_prefill_ws (split-KV) is expected to be
 * faster than fa_prefill, 0 if not, a negative fa_status_t on error (-1 bad
 * sizes, -6 no usable device).  The rule is the pages' split-K rule for an
 * underfilled part, applied to the KV dimension (page "mate: Marlin-class
 * W4A16 GEMM for mp_31 (SQMMA int4 x fp16) - #6", section "Split-K: the
 * decode occupancy lever": split when the tiles cannot cover the part, but
 * only when each piece keeps enough work to pay for the merge): split when
 * the one-shot grid (query-tile pairs) covers at most half of the SMs and the
 * longest query tile walks at least 8 KV tiles.  Queries the device's SM
 * count once (cached); launches nothing.
 */
int fa_split_kv_advised(int B, int Hq, int Hkv, int Sq, int Skv, int causal);

/*
 * fa_split_kv_advised_hd -- fa_split_kv_advised for a known head width hd
 * (the same returns; -FA_ERR_UNSUPPORTED for an hd no kernel takes; 0 for hd
 * over 128, which split-KV does not take).  Besides the underfilled-grid rule
 * above it advises split-KV for heads up to 64 wide when there are more
 * query-tile pairs than SMs but the one-shot grid's waves leave SMs idle: the
 * pairs run longest first in waves of one per SM, each wave as long as its
 * longest pair, and when the pairs' KV steps fill less than 85 % of
 * SMs x that time, the split-KV schedule's equal stream-K ranges (run by the
 * persistent kernel) finish sooner.  That is the page's split-K rule again --
 * split when the tiles cannot cover the part evenly -- for a grid of more
 * pairs than SMs (e.g. 160 equal pairs on 152 SMs fill 53 %; the chunked
 * prefill's 256 pairs fill 84 %).  Host-only; launches nothing.
 */
int fa_split_kv_advised_hd(int B, int Hq, int Hkv, int Sq, int Skv, int hd, int causal);

/*
 * fa_prefill_kvcache -- attention over a K/V cache, the read side of a
 * chunked prefill.  q, o as in fa_prefill; k_cache, v_cache are
 * [B][kv_cap][Hkv][hd] 16-bit, device, of which rows [0, kv_len) of each
 * sequence hold keys and values.  The Sq query rows are the last Sq of the
 * kv_len positions (row i sees key j iff j <= kv_len - Sq + i when causal).
 * Rows kv_len .. kv_cap - 1 never reach the result whatever they hold
 * (unwritten or stale cache memory): the TMA maps describe kv_len rows with
 * a batch stride of kv_cap rows, so rows past kv_len are loaded as zeros --
 * the pages' rule that rows at or past kv_end are zero-staged and must not
 * contribute (minfer "28 · r23 — f16-path whole-graph wall decomposition +
 * FA_TKV occupancy raise", section 3.2).
 *   bf16       0: f16 (as fa_prefill), non-zero: bfloat16
 *   workspace  NULL: the one-shot kernel; otherwise the split-KV kernel with
 *              this workspace, under fa_prefill_ws's rules for it
 * Errors: those of fa_prefill (fa_prefill_ws with a workspace), and
 * FA_ERR_INVALID_ARG for kv_len > kv_cap, a negative kv_len or kv_cap, or o
 * overlapping the caches' full kv_cap extent.
 */
int fa_prefill_kvcache(const void* q, const void* k_cache, const void* v_cache,
                       void* o, int B, int Hq, int Hkv, int Sq, int kv_len,
                       int kv_cap, int hd, int causal, float scale, int bf16,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_prefill_paged -- attention over a paged K/V cache (one-shot kernel).  q,
 * o as in fa_prefill; K and V live in pools of fixed-size pages:
 *   k_pool, v_pool  [num_blocks][page_size][Hkv][hd] 16-bit, device
 *   block_table     [B][max_pages] int32, device: key j of sequence b is row
 *                   j % page_size of pool block block_table[b][j / page_size]
 *   kv_len          keys per sequence (the same for every b); the Sq query
 *                   rows are the last Sq of them (bottom-right causal)
 *   page_size       a multiple of 128 (one KV tile never spans two pages)
 *   bf16            0: f16, non-zero: bfloat16
 * Rows of the last page past kv_len never contribute (they load as zeros).
 * A block-table entry outside [0, num_blocks) is reported in the device
 * status word (fa_debug_status() code 33) and its page reads as zeros.  The
 * pages read K/V through one contiguous row index (kv_end, the query's
 * absolute position: minfer "28 · r23 — f16-path whole-graph wall
 * decomposition + FA_TKV occupancy raise", section 3.2); the page
 * indirection is this library's extension of that index.
 * Errors: those of fa_prefill, and FA_ERR_INVALID_ARG for a page_size that is
 * not a positive multiple of 128, max_pages * page_size < kv_len,
 * num_blocks < 1, a NULL block table (kv_len > 0), or o overlapping a pool or
 * the table; FA_ERR_ALIGNMENT for a block table not 4-byte aligned.
 */
int fa_prefill_paged(const void* q, const void* k_pool, const void* v_pool,
                     const void* block_table, void* o, int B, int Hq, int Hkv,
                     int Sq, int kv_len, int hd, int page_size, int max_pages,
                     int num_blocks, int causal, float scale, int bf16,
                     void* stream);

/*
 * fa_prefill_paged_ws -- fa_prefill_paged computed by the split-KV kernel
 * (fa_prefill_ws's kernel, with the same paged producer): the arguments of
 * fa_prefill_paged, then a workspace under fa_prefill_ws's rules (caller-owned,
 * >= fa_workspace_bytes(hd), 256-byte aligned, not shared by overlapping
 * calls).  For a chunk over a long paged context,
 * where the one-shot grid leaves most SMs idle (fa_split_kv_advised).
 * Errors: those of fa_prefill_paged and fa_prefill_ws (NULL, small or
 * misaligned workspace); heads up to 128 wide.
 */
int fa_prefill_paged_ws(const void* q, const void* k_pool, const void* v_pool,
                        const void* block_table, void* o, int B, int Hq,
                        int Hkv, int Sq, int kv_len, int hd, int page_size,
                        int max_pages, int num_blocks, int causal, float scale,
                        int bf16, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * fa_kv_append -- the K/V-cache append before a chunked prefill's attention
 * (the pages' store_kv kernel, minfer "11 · P5 — prefill gap session: TM=128
 * big tiles + FA rewrite", section 3.2), for K and V in one launch:
 *     k_cache[b][positions[b][t]][h][:] = round16(k_new[b][t][h][:])
 * and the same for V, round16 being IEEE round to nearest, ties to even, into
 * f16 (bf16 == 0) or bfloat16 (bf16 != 0): values past the largest finite
 * 16-bit value become +-inf, NaN stays NaN.
 *   k_new, v_new      [B][T][Hkv][hd] f32, device, read-only, 16-byte aligned
 *   positions         [B][T] int32, device, read-only: each token's cache row
 *   k_cache, v_cache  [B][kv_cap][Hkv][hd] 16-bit, device, 16-byte aligned;
 *                     only the rows named by positions are written
 *   hd                any positive multiple of 8
 * A position outside [0, kv_cap) is skipped (nothing written for that token)
 * and reported in the device status word: fa_debug_status() returns code 32
 * with the flat index b * T + t of one such token in bits 8-31.  Positions
 * within a sequence should be distinct; of two tokens naming one row, either
 * may win.  Asynchronous on `stream` like the attention entry points.
 * Errors: FA_ERR_INVALID_ARG (null pointer, negative B or T, Hkv < 1,
 * kv_cap < 1, caches overlapping each other or the inputs),
 * FA_ERR_UNSUPPORTED (hd not a positive multiple of 8, or more than about
 * 2^31 8-element groups), FA_ERR_ALIGNMENT, FA_ERR_DEVICE, FA_ERR_LAUNCH.
 * B == 0 or T == 0 is a no-op returning FA_OK.
 */
int fa_kv_append(const void* k_new, const void* v_new, const void* positions,
                 void* k_cache, void* v_cache, int B, int T, int Hkv, int hd,
                 int kv_cap, int bf16, void* stream);

/* Size of the library's static device scratch array (one per device the
 * library runs on): 40 MiB, about 0.015 % of a 288 GB GB300. */
#define FA_STATIC_SCRATCH_BYTES (40u * 1024u * 1024u)

/*
 * fa_prefill_ws_static -- fa_prefill_ws with no caller workspace and no
 * allocation.  The pages have no counterpart to this entry point (their
 * kernel keeps no scratch); it is for callers that cannot allocate device
 * memory when they call:
 *   - an engine whose device memory is laid out once at start-up and may not
 *     grow per request: an allocation under peak load can fail or stall on
 *     the allocator, and would break the fixed layout;
 *   - a C host with no device allocator of its own, holding only the tensors
 *     it is given.
 * Same split-KV kernels and schedule as fa_prefill_ws; the scratch (m and
 * l, partial O) is a file-scope device array of FA_STATIC_SCRATCH_BYTES
 * inside the library.  Neither the call nor the library allocates or frees
 * device memory.
 *
 * Arguments: the first 12 of fa_prefill, then
 *   bf16    0: f16 Q/K/V/O (as fa_prefill); non-zero: bfloat16 (as fa_prefill_bf16)
 *   stream  cudaStream_t to enqueue on (NULL = legacy default stream)
 * Scratch need: 1048576 + pieces * 1024 * hd bytes, pieces being the
 * workspace slots of the call's schedule (at most twice its CTAs, which are
 * at most the SM count and at most 256).  A call that needs more than
 * FA_STATIC_SCRATCH_BYTES returns FA_ERR_SCRATCH and launches nothing; on a
 * 152-SM GB300 every call fits (at most 40763392 bytes, hd 128).
 * Set-up: the first call on each device looks up the array's address
 * (cudaGetSymbolAddress); nothing in it needs initialising.  Later calls only
 * launch the kernels.
 * Concurrency: every call on a device uses the same array, so calls that
 * overlap on the GPU (issued on different streams, or from several host
 * threads, without ordering between them) race and corrupt each other's
 * output.  Issue them in order, e.g. on one stream.
 * Errors: those of fa_prefill; FA_ERR_SCRATCH as above; FA_ERR_DEVICE or
 * FA_ERR_LAUNCH if the set-up fails (it is retried by the next call).
 */
int fa_prefill_ws_static(const void* q, const void* k, const void* v, void* o,
                         int B, int Hq, int Hkv, int Sq, int Skv, int hd,
                         int causal, float scale, int bf16, void* stream);

/* A static, human-readable name for a status code (never NULL). */
const char* fa_status_string(int status);

/*
 * fa_smem_bytes -- the dynamic shared memory one CTA of the kernel requests
 * for head dimension hd (that of the 64-, 128- or 256-column kernel the head
 * runs on), computed from the kernel's own tile
 * layout (Q tile, K/V stage ring, P tile, barriers, alignment slack).  Returns
 * 0 for an unsupported hd.  Host-only; no device is touched.  Exposed so the
 * launcher's request can be checked against the layout, the failure class of
 * minfer "49 · r46 (FAP1)", section 2.5 (a launcher formula that silently
 * over-requests shared memory).
 */
unsigned int fa_smem_bytes(int hd);

/*
 * fa_debug_status -- the kernel watchdog word of the current device: 0 when
 * no kernel has reported a problem since the last clear, otherwise a code
 * (bits 0-7: which wait gave up, 1 to 11 or 13 (a CTA pair's load forwarder)
 * -- or 12, a split piece the schedule gave no workspace slot (not expected),
 * 17, a persistent kernel whose shared memory was not 1024-byte aligned
 * (nothing run; not expected), 32, a cache-append position
 * out of range (fa_kv_append), or 33, a block-table entry outside the pool
 * (fa_prefill_paged); bits 8-31: the CTA or token index, saturated).  A
 * pipeline wait that does not complete within the watchdog limit records its
 * code here, makes its CTA skip its remaining work and exit cleanly (no trap),
 * so the context stays usable.  Synchronises the device.  Returns -1 if the
 * word cannot be read.
 */
int fa_debug_status(void);

/* Reset the watchdog word of the current device to 0 (synchronous). Returns an fa_status_t. */
int fa_debug_status_clear(void);

/*
 * fa_debug_set_watchdog_ns -- a testing hook: the limit, in nanoseconds, that
 * each pipeline wait of the kernels launched after this call may take before
 * its CTA gives up (default 2 s; 0 restores it).  A tiny limit makes waits run
 * out on purpose, so a test can check that a CTA which gives up records its
 * code in the watchdog word, waits for the copies and MMAs it already issued,
 * frees its TMEM and exits, and that the context stays usable.  The output of
 * a call whose CTAs gave up is undefined.  Host-only (no device call);
 * process-wide.  Returns FA_OK.
 */
int fa_debug_set_watchdog_ns(unsigned long long ns);

/*
 * fa_debug_force_path -- a testing and measurement hook: the kernel that calls
 * made after it run on, process-wide.  0: the library's own choice (the
 * default); 1: the one-shot kernel, also for calls given a workspace (no
 * split); 2: the persistent kernel -- over whole query-tile pairs, each CTA
 * taking pairs in snake order, for calls without a workspace, and for every
 * split-KV schedule (not only multi-segment ones) for calls with one; 3: the
 * CTA-pair kernel (two CTAs on two SMs per unit of four query heads, paired
 * tcgen05 MMAs with M = 256) for the calls it applies to -- contiguous K/V,
 * GQA groups of a multiple of 4 query heads, heads 72 to 128 wide, no
 * workspace -- and the library's choice for the others.  (Path 3 measured
 * slower than the library's choice; it is kept for measurement.)  Heads
 * wider than 128 always run on the one-shot kernel.  The result is the same
 * within the parity tolerance whatever the path.  Host-only.  Returns FA_OK,
 * or FA_ERR_INVALID_ARG for another value (nothing changed).
 */
int fa_debug_force_path(int path);

/*
 * fa_debug_schedule -- the work split fa_prefill_ws launches for a shape on
 * a GPU of `sms` SMs (host-only, no device call; for tests and tools).  The
 * query-tile pairs ("pairs") are numbered like the one-shot grid, longest
 * first.  CTA c starts at pair cta_pair[c], KV step cta_step[c], and ends
 * where CTA c+1 starts; entry [ctas] is the end (pair count, step 0).
 *   cta_pair, cta_step   host arrays of at least 257 ints (written)
 *   pair_steps           host array of at least max_pairs ints receiving
 *                        each pair's KV steps, or NULL
 *   out                  host array of 4 ints (written): CTAs, 1 if every
 *                        CTA runs a single segment (no more pairs than CTAs:
 *                        each pair cut into near-equal pieces), pairs split
 *                        between CTAs (merged by the second kernel), piece
 *                        slots used in the workspace
 * Returns the number of pairs (>= 0), -FA_ERR_INVALID_ARG for a bad shape,
 * sms < 1 or a NULL array, -FA_ERR_UNSUPPORTED when pair_steps is given and
 * there are more than max_pairs pairs.
 */
int fa_debug_schedule(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int sms,
                      int* cta_pair, int* cta_step, int* pair_steps, int max_pairs,
                      int* out);

/*
 * fa_debug_row_pairing -- which query tile of a head the one-shot grid leaves
 * without a partner, for a shape on a GPU of `sms` SMs (host-only, no device
 * call; for tests and tools).  It matters for row pairs (MHA or an odd GQA
 * group: a CTA holds two adjacent 128-row tiles of one head) with an odd tile
 * count.  Under the causal mask tile 0 sees the fewest keys and the last tile
 * the most; a CTA's time follows its KV steps, and one tile alone walks them
 * little faster than a pair.  So leaving tile 0 alone cuts the grid's total
 * steps, while near one wave the longest CTA sets the time and the last tile
 * alone is shorter than a pair there.  The library takes the pairing that a
 * list-scheduling model of the grid expects to finish first; the split-KV
 * paths always leave tile 0 alone (their ranges even out the lengths).
 * Returns 1 when tile 0 goes alone (then pairs (2p - 1, 2p)), 0 when the last
 * tile does (pairs (2p, 2p + 1)) or no tile goes alone (head pairs, even tile
 * counts, one tile), -FA_ERR_INVALID_ARG for a bad shape or sms < 1.
 */
int fa_debug_row_pairing(int B, int Hq, int Hkv, int Sq, int Skv, int causal, int sms);

#ifdef __cplusplus
}
#endif

#endif /* FA_PREFILL_H */

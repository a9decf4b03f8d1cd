/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) single-token MLA decode library.
 *
 * Operation (amd-mixed-mla submission 599694, `_bmm` path; geometry and sm_scale from
 * the module constants of submissions 727205 / 700955 / 599694):
 *   16 query heads share one latent KV head of width 576 (512 "nope" + 64 rope).
 *   For batch row b, head h, over cached rows r in [kv_indptr[b], kv_indptr[b+1]):
 *     s_r      = (1/sqrt(576)) * q[b,h,:] . Khat_r          Khat_r = dequantised row r
 *     out[b,h] = sum_r softmax(s)_r * Khat_r[0:512]          (V = first 512 columns)
 *   Page size 1: row index = token index, rows of one sequence are contiguous.
 *
 * Method: split-KV flash decoding (submission 727205 `mla_s1` + `mla_rd`, submission
 * 700955 `mla_attn_v71` + `reduce_lse_v71`, submission 599694 `_flash_fp8_split_s1/_s2`):
 * each sequence's rows are cut into splits, each split produces an online-softmax
 * partial result (normalised output + log-sum-exp), and the partials are merged by
 * log-sum-exp weights.  Here the merge runs inside the same kernel: the CTA that writes
 * a sequence's last partial merges all of them, so one call is one kernel launch.
 *
 * All pointers are DEVICE pointers unless stated otherwise.  The caller owns every
 * buffer it passes; the library never frees or retains them past the call.  Calls are
 * asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream): the
 * library performs no host synchronisation and never reads device data on the host.
 * Every entry point returns an mla_status (0 = success).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_NUM_HEADS 16
#define MLA_HEAD_DIM 576
#define MLA_V_DIM 512
#define MLA_MX_BLOCK 32
#define MLA_MX_PACKED_BYTES 288 /* bytes of e2m1 nibbles per cached row */
#define MLA_MX_SCALES 18        /* e8m0 scales per cached row */

/* KV-cache storage encodings.
 *  BF16     : kv = bf16 [T][576].
 *  FP8_E4M3 : kv = e4m3fn codes uint8 [T][576]; value = code * kv_scale[0] (one fp32 per
 *             tensor; submission 599694 fp8 flash-decode dequantises this way).
 *  MXFP4    : kv = uint8 [T][288], element 2i in the low nibble of byte i and 2i+1 in the
 *             high nibble (submission 700955 `mla_attn_v74`); kv_scale = uint8 [T][18]
 *             e8m0 block scales (value = e2m1 * 2^(E-127), one scale per 32 elements). */
typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1, MLA_KV_MXFP4 = 2 } mla_kv_dtype;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1, /* a host-side argument check failed; nothing was launched */
  MLA_ERR_UNSUPPORTED = -2, /* device is not sm_103 / lacks the shared memory this needs */
  MLA_ERR_CUDA = -3,        /* a CUDA runtime/driver call or a launch failed */
  MLA_ERR_NO_MEMORY = -4,   /* the library's partial-result workspace could not grow */
  MLA_ERR_TIMEOUT = -5      /* a kernel pipeline wait ran past its limit (device status) */
} mla_status;

/*
 * mla_decode -- out[b,h,:] for every batch row b and head h.
 *
 *  q          bf16 [batch][16][576], contiguous, 16-byte aligned.
 *  kv         cache rows, layout per kv_dtype above, contiguous, 16-byte aligned.
 *  kv_scale   NULL for BF16; const float* [1] (device) for FP8_E4M3; const uint8_t*
 *             [T][18] (device, row stride 18 bytes) for MXFP4.
 *  kv_indptr  int32 [batch+1] (device): kv_indptr[0] = 0, non-decreasing, and every
 *             kv_indptr[b+1] <= T (the number of rows in kv).  The library reads only
 *             rows inside these ranges.  A violation is undefined behaviour (the library
 *             cannot check device data without a host sync).
 *  out        bf16 [batch][16][512] (device), written; 4-byte aligned.
 *  batch      >= 1.
 *  num_splits >= 1: cut every sequence into that many splits (BN = 128-token-rounded
 *             chunks, submission 727205 `mla_s1` split rule; splits past the end are
 *             empty; num_splits = 1 writes out directly with no merge).
 *             <= 0: the library balances the batch over the GPU's SMs (one persistent CTA
 *             per SM, contiguous token ranges that may span several sequences) and merges
 *             the pieces of each sequence.  The ranges split the batch's cost evenly: its
 *             tokens plus, for every sequence start after the first, the rows a CTA gets
 *             through in the time it loses moving to the next sequence (the split model's
 *             x of mla_decode_pick_splits: 521 fp8 rows, 260 bf16 rows, 294 MXFP4 rows),
 *             so that a CTA that crosses
 *             sequence boundaries is given fewer tokens.
 *             At most 4096 splits.  mla_decode_pick_splits returns a good value.
 *  kv_dtype   an mla_kv_dtype value.
 *  stream     cudaStream_t or NULL.
 * Empty sequences (kv_indptr[b] == kv_indptr[b+1]) produce zeros.
 * Errors: MLA_ERR_INVALID_ARG before any launch for null/misaligned pointers, batch <= 0,
 * an unknown kv_dtype or num_splits > 4096; MLA_ERR_UNSUPPORTED if the current device is
 * not compute capability 10.3; MLA_ERR_NO_MEMORY if the workspace cannot grow;
 * MLA_ERR_CUDA if a launch fails (the CUDA error is cleared and its name is available
 * from mla_last_cuda_error()).
 * The partial-result workspace is library-owned (one per device, grow-only).  A call
 * holds the library's workspace mutex from the workspace check until its kernel is
 * enqueued, and a grow synchronises the device before it frees the old buffers, so
 * concurrent calls from several host threads never see a freed buffer.  The kernels of
 * every call on a device share that one workspace, though: two calls whose kernels may
 * overlap on the GPU (different streams with no ordering between them) race on its
 * partial results and piece counters and may return wrong results.  Order such calls
 * (one stream, or events).
 */
int mla_decode(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_indptr,
               void* out, int batch, int num_splits, int kv_dtype, void* stream);

/*
 * mla_decode_paged -- the same decode over a paged KV cache: the pages of a sequence need
 * not be contiguous or in order.  Layout of the page table as in the library-routed a16w8
 * path of amd-mixed-mla submission 700955 (a page-level indptr, `kv_indices`,
 * `kv_last_page_len`, `page_size`); the operation on each sequence is exactly mla_decode's.
 *
 *  kv               cache rows grouped in pages of page_size rows: physical page P holds
 *                   rows [P * page_size, (P + 1) * page_size) of the same row layout as
 *                   mla_decode (bf16 [.][576], e4m3 [.][576] or MXFP4 [.][288]); 16-byte aligned.
 *  kv_scale         as mla_decode; for MXFP4 indexed by the same (physical) row.
 *  kv_page_indptr   int32 [batch+1] (device): sequence b's pages are
 *                   kv_page_indices[kv_page_indptr[b] .. kv_page_indptr[b+1]).
 *  kv_page_indices  int32 (device): physical page numbers, in sequence order.
 *  kv_last_page_len int32 [batch] (device): rows used in the sequence's last page,
 *                   1 .. page_size (ignored for a sequence with no pages, which has length 0).
 *                   Sequence b has (npages_b - 1) * page_size + kv_last_page_len[b] tokens.
 *  page_size        1, 2, 4, 8, 16, 32, 64 or 128.  Pages of 8 rows and more are loaded one
 *                   TMA box per page; pages of 1, 2 or 4 rows (fewer than a box's 8-row swizzle
 *                   atom; the pages' persistent default is 2) four rows per TMA gather (bf16,
 *                   fp8) or 16 bytes at a time (MXFP4).
 *  num_splits       as mla_decode.  In the balanced mode (<= 0) the token positions are
 *                   those of the page space (sequence b starts at kv_page_indptr[b] *
 *                   page_size; the unused rows of its last page belong to no CTA's work)
 *                   and the CTAs' cut points, which split the token count evenly (no
 *                   crossing cost), are rounded down to multiples of 128, so that every
 *                   128-token tile starts on a page boundary.
 * Every page number times page_size plus page_size must be a row inside kv, and every
 * index read must lie inside kv_page_indices; violations are undefined behaviour, as with
 * kv_indptr.  Errors: as mla_decode, plus MLA_ERR_INVALID_ARG for a page_size that is not
 * a power of two in [1, 128] or a null page table.
 */
int mla_decode_paged(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_page_indptr,
                     const int32_t* kv_page_indices, const int32_t* kv_last_page_len, int page_size, void* out,
                     int batch, int num_splits, int kv_dtype, void* stream);

/*
 * mla_decode_paged_multi -- mla_decode_paged with several query tokens per sequence (the
 * q_len > 1 form of the paged decode interface: the `qo_indptr` argument of the a16w8 path
 * of amd-mixed-mla submission 700955, which the pages only call with one token per
 * sequence).  The q_len_b = qo_indptr[b+1] - qo_indptr[b] new tokens of sequence b are the
 * last q_len_b tokens of its cache (their keys and values already appended), and each sees
 * the cache up to and including itself: query row qo_indptr[b] + t (0 <= t < q_len_b)
 * attends to the first L_b - q_len_b + 1 + t cached tokens of sequence b (none if that is
 * <= 0, which gives zeros).  Every (row, head) is otherwise exactly mla_decode's operation.
 *
 *  q            bf16 [total_q][16][576] (device), 16-byte aligned; rows grouped by sequence.
 *  qo_indptr    int32 [batch+1] (device): qo_indptr[0] = 0, non-decreasing,
 *               qo_indptr[batch] = total_q (a violation is undefined behaviour).
 *  total_q      >= 1: query rows.
 *  out          bf16 [total_q][16][512] (device).
 *  batch        >= 1: sequences (entries of the page table).
 *  num_splits   >= 1: uniform splits of the visible range; <= 0: the library's choice,
 *               max(1, floor(SMs / U)) uniform splits (no balanced mode), U = ceil(total_q / 2)
 *               for bf16 and fp8 caches, total_q for MXFP4.
 *  kv, kv_scale, kv_page_indptr, kv_page_indices, kv_last_page_len, page_size, kv_dtype,
 *  stream: as mla_decode_paged.
 * bf16 and fp8 caches: the query tokens of a sequence are decoded two at a time (tokens 2i
 * and 2i + 1 share one pass over the cache; the 32 query rows x heads sit on the MMA's N
 * side and each keeps its own causal mask).  MXFP4 caches: each query row reads its own
 * visible range (rows of one sequence share the cache through L2).  Errors: as
 * mla_decode_paged, plus MLA_ERR_INVALID_ARG for a null or misaligned qo_indptr or
 * total_q <= 0.
 */
int mla_decode_paged_multi(const void* q, const int32_t* qo_indptr, int total_q, const void* kv,
                           const void* kv_scale, const int32_t* kv_page_indptr,
                           const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                           int page_size, void* out, int batch, int num_splits, int kv_dtype,
                           void* stream);

/*
 * mla_decode_pick_splits -- host-only choice of num_splits for mla_decode on a batch of
 * `batch` sequences of about kv_len_hint tokens each, on a GPU with num_sms SMs.
 * The split model of amd-mixed-mla submission 700955 (`_compute_custom_splits`: utilisation
 * of the CTA slots times L / (L + per-split overhead)), with this kernel's own costs counted
 * in cache rows (a row = the bytes of one cached token: 1152 bf16, 576 fp8, 306 MXFP4, which
 * is why kv_dtype is an argument; an MXFP4 CTA is bound by its dequantisation at 0.30 of the
 * HBM rate, measured, so an MXFP4 row counts 306 / 0.30 bytes below):
 *   c = 32,832 / row   one piece (16 x 513 fp32 partial output and log-sum-exp), written once
 *                      and read once by the CTA that merges the sequence's ns pieces;
 *   w = 222,000 / row  one wave of CTAs: a CTA's start-up and final drain (about 2 + 3 us,
 *                      measured) times one SM's share of the HBM bandwidth (6.76 TB/s / 152);
 *   x = 300,000 / row  a CTA moving from one sequence to the next in the balanced mode (the
 *                      pipeline drain and refill: about 6.7 us, measured, times the same share).
 * Time of the slowest CTA, in rows, with B = batch, L = kv_len_hint, S = num_sms:
 *   uniform ns (1 <= ns <= ceil(L / 128)):  waves * (chunk + w + c) + ns * c   (no c terms for ns = 1),
 *     waves = ceil(B ns / S), chunk = ceil(L / ns) rounded up to 128-row tiles;
 *   balanced: R + w + s c + (s - 1) x + p c,  R = B L / S, s = ceil(R / L) + 1, p = ceil(L / R) + 1.
 * Returns the uniform ns of least time (the smallest on ties), or 0 (the balanced mode) when
 * that is faster.  The hint describes a batch of equal lengths; for a batch whose lengths
 * vary widely call mla_decode with num_splits <= 0 (the balanced mode) directly.
 * Returns MLA_ERR_INVALID_ARG for batch <= 0, kv_len_hint < 0, num_sms <= 0 or an unknown
 * kv_dtype.
 */
int mla_decode_pick_splits(int batch, int kv_len_hint, int num_sms, int kv_dtype);

/* Number of partial-result slots a call with these arguments needs (for sizing). */
int mla_decode_workspace_slots(int batch, int num_splits, int num_sms);

/* Grows the current device's workspace so that calls needing up to `slots` partial slots
 * allocate nothing (useful before timing or graph capture).  Returns an mla_status. */
int mla_decode_reserve_workspace(int slots);

/* Frees the library's workspace on the current device (synchronises the device). */
int mla_decode_release_workspace(void);

/* Reads and (if clear != 0) resets the current device's kernel status word.  Synchronises
 * the device.  Returns MLA_OK, or MLA_ERR_TIMEOUT if a pipeline wait in a kernel gave up
 * since the last clear.  After a timeout the output of that call is undefined and the
 * workspace's piece counters may be left non-zero: call mla_decode_release_workspace
 * before the next call that splits sequences. */
int mla_decode_device_status(int clear);

/* Sets the time after which a kernel's pipeline wait gives up, sets the status word and
 * lets the kernel return (default 2e9 ns).  For tests of the failure path.  The waits a CTA
 * makes for its own copies and MMAs in flight before it exits keep a fixed 2 s limit. */
void mla_decode_set_wait_limit_ns(unsigned long long ns);

/* Test hook (failure path without a fault): while on != 0, every mla_decode call's QK
 * issuer first waits on a barrier that nothing completes, so that the wait runs past the
 * limit, the device status reads MLA_ERR_TIMEOUT and the kernel returns.  Never set outside
 * tests; mla_decode_noalloc ignores it. */
void mla_decode_set_test_stall(int on);

/* Test hook: the crossing cost, in cache rows, that the balanced mode of mla_decode and
 * mla_decode_noalloc charges per sequence start when it cuts the batch (rows >= 0; a large
 * value leaves CTAs whose range lies inside one crossing, with no work).  rows < 0 restores
 * the default, x of the split model (mla_decode_pick_splits) for the call's cache dtype. */
void mla_decode_set_cross_rows(int rows);

/* Timing hooks.  Between begin and end, every mla_decode call records CUDA events on its
 * stream around its split kernel and around the whole call.  end() waits for those events
 * and returns the summed split-kernel time, the summed call time (ms) and the number of
 * calls recorded, then stops recording.  Returns an mla_status. */
int mla_decode_profile_begin(void);
int mla_decode_profile_end(double* split_ms, double* call_ms, int* calls);

/*
 * mla_decode_noalloc -- the same decode as mla_decode, with the same arguments, for callers
 * that must not allocate device memory on the decode path (a serving engine or plugin host
 * whose own pool owns every device allocation, or a latency-critical loop that cannot
 * afford cudaMalloc / cudaFree, the latter synchronising the whole device).  The pages
 * have no counterpart: this is a deployment variant of mla_decode.
 *
 * Scratch (split partial results, the per-sequence piece counters that select the
 * merging CTA, and the kernel status word) lives in a fixed array
 * inside the library's device code instead of a cudaMalloc'd workspace: every GPU that
 * loads the library holds it (about MLA_NOALLOC_MAX_SLOTS x 32.8 KB, 16.8 MB) until the
 * process exits.  The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *  - Limit: the call needs batch*num_splits partial slots (num_splits >= 2), none
 *    (num_splits == 1), or batch + SMs - 1 (num_splits <= 0); more than
 *    MLA_NOALLOC_MAX_SLOTS returns MLA_ERR_NO_MEMORY before any launch.
 *  - The first call on each device (with that device current) looks up the array's device
 *    address once (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - All calls share the one array, which keeps the previous call's contents.  Every call
 *    first clears, with one stream-ordered memset on `stream`, the status word and the
 *    piece counters it uses, so a call that a pipeline timeout cut short leaves nothing
 *    behind for the next one.  Calls that overlap on the GPU (different streams with no
 *    ordering between them) race on the array: serialise them on one stream or order
 *    them with events.
 *  - A pipeline timeout (the limit set by mla_decode_set_wait_limit_ns) is recorded in
 *    the array's own status word: read it with mla_decode_noalloc_status after the call
 *    and before the next one (the next call clears it).
 * Errors as mla_decode, plus MLA_ERR_NO_MEMORY when the scratch is too small.
 */
#define MLA_NOALLOC_MAX_SLOTS 512
int mla_decode_noalloc(const void* q, const void* kv, const void* kv_scale, const int32_t* kv_indptr,
                       void* out, int batch, int num_splits, int kv_dtype, void* stream);

/* Status of the most recent mla_decode_noalloc call on the current device: waits for the
 * device (cudaMemcpy), returns MLA_OK or MLA_ERR_TIMEOUT, and resets the word if
 * clear != 0.  Allocates nothing. */
int mla_decode_noalloc_status(int clear);

/* Static string for a status code; never NULL. */
const char* mla_status_string(int status);

/* Name of the last CUDA error the library saw on this thread ("" if none). */
const char* mla_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */

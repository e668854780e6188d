/*
 * bd_attn.h -- C ABI of libbd: block-causal (per-document) varlen attention
 * over packed multi-document sequences, computed one contiguous
 * context-parallel query chunk at a time, for sm_103a (GB300).
 *
 * What the operation is (NeMo Automodel page "block-diagonal varlen CP for
 * packed sequences"):
 *   - documents are packed back to back into one sequence of S rows, their
 *     boundaries given as cumulative lengths cu_seqlens (Summary);
 *   - attention is block-causal per document: row i sees row j iff both lie in
 *     the same document and j <= i; nothing leaks across a document boundary
 *     (Motivation; Key correctness property 1);
 *   - S is padded to a multiple of the context-parallel size cp and rank r owns
 *     the contiguous rows [r*L, (r+1)*L), L = S/cp (Design overview, batch.py);
 *   - a document straddling the chunk's left edge gives an asymmetric varlen
 *     segment with more keys than queries, aligned bottom-right (Key
 *     correctness property 2);
 *   - K/V reach a chunk either as the whole sequence (fused [K;V] all-gather,
 *     the default) or needed-only, starting at the first document the chunk
 *     overlaps (Summary; Design overview, exchange.py);
 *   - the backward of the all-gather is a reduce-scatter SUM: per-chunk dK/dV
 *     partials add up at the rows' owner (Design overview, exchange.py);
 *   - every index a varlen kernel consumes is validated on the host first,
 *     because a bad offset is an asynchronous illegal memory access, not an
 *     error (Key correctness property 4).
 *
 * Conventions for every call:
 *   - Return value: BD_OK (0) or a negative bd_status. Nothing is launched
 *     when a call fails validation. bd_last_error() gives a message for the
 *     calling thread's last failure.
 *   - Ownership: the caller allocates every buffer (host plan, device plan,
 *     tensors, workspace). The library keeps no device allocation of its own.
 *   - Device calls are asynchronous and ordered on the given cudaStream_t
 *     (passed as void*; NULL is the legacy default stream). They do no host
 *     synchronisation.
 *   - Softmax scale is 1/sqrt(d); LSE is the natural-log log-sum-exp of the
 *     scaled scores, in fp32. Padding rows (>= cu_seqlens[last]) get O = 0,
 *     LSE = -inf and zero gradients. GQA maps query head h to key/value head
 *     h / (H / Hkv).
 */
#ifndef BD_ATTN_H
#define BD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BD_API __attribute__((visibility("default")))
#else
#define BD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BD_OK = 0,
  BD_ERR_ARG = -1,            /* NULL pointer, bad size or bad enum value        */
  BD_ERR_CU_SEQLENS = -2,     /* cu_seqlens[0] != 0, decreasing, or > S          */
  BD_ERR_NOT_DIVISIBLE = -3,  /* S % cp != 0: pad S first (bd_padded_len)        */
  BD_ERR_RANK = -4,           /* rank outside [0, cp)                            */
  BD_ERR_CAPACITY = -5,       /* output array or workspace too small             */
  BD_ERR_ALIGN = -6,          /* pointer/stride not 16-byte aligned, d not unit  */
  BD_ERR_UNSUPPORTED = -7,    /* head dim, head ratio or layout not supported    */
  BD_ERR_CUDA = -8,           /* a CUDA runtime/driver call failed               */
  BD_ERR_DEVICE_TIMEOUT = -9, /* a kernel gave up waiting and stopped early      */
  BD_ERR_PLAN = -10           /* plan blob corrupt or built for other shapes     */
} bd_status;

typedef enum {
  BD_KV_GATHER = 0, /* K/V buffer row j = global row j (fused all-gather)            */
  BD_KV_WINDOW = 1  /* K/V buffer of chunk c starts at global row kv_start of c     */
} bd_kv_mode;

/* One varlen segment of a chunk, in global rows. The segment's queries are
 * [q_start, q_start+q_len); its keys are [k_start, k_start+k_len) with
 * k_start = start of document `doc` and k_start+k_len = q_start+q_len. Local
 * query i (0-based in the segment) sees local key j iff j <= i + diag_off,
 * diag_off = k_len - q_len (bottom-right alignment). */
typedef struct {
  int32_t doc, q_start, q_len, k_start, k_len, diag_off;
} bd_segment_t;

/* Per-chunk header. row_offset = rank*L. s_valid = cu_seqlens[ndocs]. n_pad =
 * rows of the chunk at or past s_valid. [kv_start, kv_end) = the needed-only
 * key window: kv_start = start of the first document the chunk overlaps,
 * kv_end = min(row_offset + L, s_valid); for an all-padding chunk both equal
 * min(row_offset, s_valid) and nseg = 0. */
typedef struct {
  int32_t S, cp, rank, L, row_offset, s_valid, n_pad, kv_start, kv_end, nseg;
} bd_chunk_hdr;

/* bd_segment -- varlen metadata of chunk `rank` of `cp` for one packed sequence:
 * the contiguous rows [rank*L, (rank+1)*L) (NeMo Automodel page "block-diagonal
 * varlen CP for packed sequences", Design overview, batch.py), cut into one
 * segment per document they overlap (Design overview, kernels.py), a document
 * straddling the left edge giving more keys than queries with bottom-right
 * alignment (Key correctness property 2), every index validated here on the
 * host (Key correctness property 4).
 *   cu_seqlens  host int32[ndocs+1], cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[ndocs] <= S. Zero-length documents are allowed and
 *               produce no segment.
 *   S           padded sequence length, S % cp == 0.
 *   hdr         host output header (required).
 *   segs        host output array of seg_capacity entries, or NULL to only
 *               count (hdr->nseg is always set).
 * Errors: BD_ERR_ARG, BD_ERR_CU_SEQLENS, BD_ERR_NOT_DIVISIBLE, BD_ERR_RANK,
 * BD_ERR_CAPACITY (segs non-NULL and seg_capacity < nseg; hdr still valid).
 * Pure host function: same inputs, same bytes out. */
BD_API int32_t bd_segment(const int32_t* cu_seqlens, int32_t ndocs, int32_t S, int32_t cp,
                   int32_t rank, bd_chunk_hdr* hdr, bd_segment_t* segs,
                   int32_t seg_capacity);

/* Smallest multiple of cp that is >= s (the padding step of batch.py). */
BD_API int32_t bd_padded_len(int32_t s, int32_t cp);

/* bd_doc_ids_to_cu -- cu_seqlens from a 1-D per-token document-id array (the
 * page's "1-D document ids" input, NeMo Automodel page "block-diagonal varlen
 * CP for packed sequences", Proof). doc_ids: host int32[n]; a document is a
 * maximal run of equal ids; ids must be non-decreasing over the valid tokens;
 * negative ids mark padding and may only form a suffix. Writes ndocs+1 entries
 * to cu_out (cap entries available) and ndocs to *ndocs_out.
 * Errors: BD_ERR_ARG, BD_ERR_CU_SEQLENS (decreasing ids, padding not a
 * suffix), BD_ERR_CAPACITY (cap too small; *ndocs_out still set). */
BD_API int32_t bd_doc_ids_to_cu(const int32_t* doc_ids, int32_t n, int32_t* cu_out, int32_t cap,
                         int32_t* ndocs_out);

/* One transfer of a needed-only K/V exchange: global rows
 * [src_row, src_row + n_rows) owned by rank src_rank land at row dst_row of
 * the receiving rank's window buffer. In the backward the same rows of the
 * window's dK/dV go back to src_rank and are added at src_row (index_add). */
typedef struct {
  int32_t src_rank, src_row, n_rows, dst_row;
} bd_xfer_t;

typedef enum {
  BD_XCHG_LOCAL = 0, /* the window lies inside the rank's own rows (or is empty) */
  BD_XCHG_HALO = 1,  /* remote rows come from the left neighbour only          */
  BD_XCHG_A2A = 2    /* remote rows come from two or more ranks (all-to-all-v) */
} bd_xchg_kind;

/* bd_exchange_plan -- the transfers that build rank `rank`'s needed-only K/V
 * window [kv_start, kv_end) from the contiguous owner slices (rank q owns rows
 * [q*L, (q+1)*L)): left-neighbour halo when a straddling document reaches back
 * one rank, all-to-all-v when it reaches further (same page, Summary; Design
 * overview, exchange.py). Transfers are in increasing src_rank order and cover
 * the window exactly once; the rank's own rows appear as a transfer from
 * itself. xfers may be NULL to count only. Errors as bd_segment, plus
 * BD_ERR_CAPACITY. */
BD_API int32_t bd_exchange_plan(const int32_t* cu_seqlens, int32_t ndocs, int32_t S, int32_t cp,
                         int32_t rank, int32_t* kind_out, bd_xfer_t* xfers, int32_t cap,
                         int32_t* nxfer_out);

/* Description of a step's work: B packed sequences of padded length S, each cut
 * into cp chunks of L = S/cp rows, of which the plan covers `nchunks` (chunk c
 * of the plan is rank ranks[c]; ranks == NULL means ranks 0..nchunks-1). One
 * plan serves one chunk (a per-rank call) or all chunks of all sequences (the
 * batched single-GPU grid). */
typedef struct {
  int32_t B, S, cp, nchunks;
  const int32_t* ranks;       /* host int32[nchunks] or NULL                      */
  int32_t H, Hkv, d;          /* d in {64, 128, 256}; H % Hkv == 0               */
  int32_t kv_mode;            /* bd_kv_mode                                       */
  const int32_t* cu_seqlens;  /* host: all sequences' cu arrays back to back      */
  const int32_t* cu_offsets;  /* host int32[B+1]: sequence b's array is
                                 cu_seqlens[cu_offsets[b] .. cu_offsets[b+1])    */
} bd_plan_desc;

/* Size in bytes of the plan blob for `desc` (validates desc like bd_segment). */
BD_API int32_t bd_plan_bytes(const bd_plan_desc* desc, size_t* bytes);

/* Build the plan blob into caller-owned host memory `blob` (16-byte aligned,
 * blob_bytes >= bd_plan_bytes). The caller copies the same bytes once per step
 * to device memory (16-byte aligned, writable: kernels record a failure status
 * in it, and forward launches take their work-unit claim counters from 8 slots
 * in it, launch after launch in turn, each slot returned to zero by the last CTA
 * of its launch) and passes both copies to the attention calls, which size their
 * launches from the host copy and read the device copy. Up to 8 forward launches
 * sharing one device copy may run at the same time (on unordered streams); a
 * ninth in flight would share a slot with the first and take units from it.
 * Backward launches keep their counters in their workspace: ones that share the
 * device plan but not the workspace may overlap. (The plan blob also holds the
 * backward's work lists; the pages' kernels.py builds the equivalent varlen
 * metadata once per step, NeMo Automodel page "block-diagonal varlen CP for
 * packed sequences", Design overview.) */
BD_API int32_t bd_plan_build(const bd_plan_desc* desc, void* blob, size_t blob_bytes);

/* Read back the header of chunk item `item` (item = b*nchunks + c) and its
 * segments from a host plan blob. */
BD_API int32_t bd_plan_chunk(const void* plan_host, int32_t item, bd_chunk_hdr* hdr,
                      bd_segment_t* segs, int32_t seg_capacity);

/* Useful (unmasked) (query, key) pairs per head over all items of a plan. */
BD_API int64_t bd_plan_useful_pairs(const void* plan_host);

/* bd_plan_set_dropout -- turn attention dropout on (p > 0) or off (p = 0) in a
 * host plan blob, before it is copied to the device. The native Flash path the
 * NeMo Automodel page forwards dropout to (Proof, GPU varlen tests) gives no
 * formulas; the reading implemented: the forward keeps probability P_ij with
 * keep_ij = (u_ij >= t), t = floor(p * 2^32 + 1/2) capped at 2^32 - 1, and
 * computes O = sum_j P_ij keep_ij v_j / (1 - p) with the undropped LSE; the
 * backward regenerates the same mask (dS_ij = P_ij (keep_ij dP_ij / (1 - p) - D_i),
 * D_i = <dO_i, O_i>). u_ij is word 2 (i mod 2) + (j mod 2) of Philox4x32-10
 * (Salmon et al., SC 2011) at counter (j / 2, i / 2, h, b) under the key
 * (seed mod 2^32, seed / 2^32); i, j are global query / key rows of sequence b
 * and h the query head. Returns BD_ERR_ARG unless 0 <= p < 1. */
BD_API int32_t bd_plan_set_dropout(void* plan_host, double p, uint64_t seed);

/* A strided device tensor whose last (head) dimension is contiguous.
 * Query-like tensors (q, out, dout, dq) are [B, nchunks, L, H, d]; key-like
 * tensors (k, v, dk, dv) are [B, Ck, rows, Hkv, d] with Ck = 1 for
 * BD_KV_GATHER (one buffer per sequence, row = global row) and Ck = nchunks
 * for BD_KV_WINDOW (one window buffer per chunk, row 0 = kv_start of that
 * chunk). Strides are in elements. `rows` is the extent of the row dimension:
 * L for query-like tensors, the buffer length for key-like ones (GATHER:
 * >= s_valid of every sequence; WINDOW: >= kv_end - kv_start of every chunk).
 * Pointers and the b/c/row/head strides (in bytes) must be 16-byte aligned. */
typedef struct {
  void* ptr;
  int64_t stride_b, stride_c, stride_row, stride_head;
  int32_t rows;
  int32_t reserved;
} bd_tensor;

/* Strided fp32 LSE / softmax-statistics tensor [B, nchunks, H, L], row dim contiguous. */
typedef struct {
  float* ptr;
  int64_t stride_b, stride_c, stride_head;
} bd_rowstat;

/* bd_attn_fwd -- forward of every chunk item in the plan: for each query row
 * of each chunk, O = softmax(scale * q K^T restricted to the row's document and
 * causal past) V and LSE -- the block-causal varlen attention of a chunk's query
 * rows against all-gathered or needed-only K/V (NeMo Automodel page
 * "block-diagonal varlen CP for packed sequences", Summary; Key correctness
 * properties 1 and 2), whose concatenation over chunks equals full attention
 * under the block-causal mask. q, k, v bf16; out bf16 (same layout rules as q);
 * lse fp32. row_offset: -1 to take every chunk's offset from the plan, or
 * the expected rank*L of a single-chunk plan (checked; BD_ERR_PLAN if it
 * differs). Rows of K/V at or past s_valid must hold finite values (they are
 * multiplied by exact zeros). */
BD_API int32_t bd_attn_fwd(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                    const bd_tensor* k, const bd_tensor* v, int32_t row_offset,
                    bd_tensor* out, bd_rowstat* lse, void* stream);

/* bd_attn_fwd_ex -- bd_attn_fwd that also sets dq_zero, an fp32 query-like
 * tensor [B, nchunks, L, H, d] (the backward's dq accumulator), to zero while
 * the forward runs: warps of the forward kernel that have no attention work
 * store the zeros, so a training step needs no separate clearing pass and the
 * backward can be told so (BD_BWD_DQ_ZEROED). dq_zero may be NULL (then this is
 * bd_attn_fwd). It must not alias q, k, v, out or lse. Errors as bd_attn_fwd,
 * plus BD_ERR_ARG / BD_ERR_ALIGN for a bad dq_zero (rows must equal L). This
 * clearing is a library addition; the NeMo Automodel page's forward has none. */
BD_API int32_t bd_attn_fwd_ex(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                       const bd_tensor* k, const bd_tensor* v, int32_t row_offset,
                       bd_tensor* out, bd_rowstat* lse, bd_tensor* dq_zero, void* stream);

/* Workspace bytes bd_attn_bwd needs for this plan: per row and head D = <dO, O>
 * and the LSE in log2 units, and the main kernel's work-unit counters (zeroed
 * by bd_attn_bwd_pre). Calls that overlap on the GPU need workspaces of their
 * own. */
BD_API int32_t bd_attn_bwd_workspace(const void* plan_host, size_t* bytes);

/* bd_attn_bwd -- backward of every chunk item in the plan for the loss
 * sum(out * dout): the analytic gradient of bd_attn_fwd, with the all-gather's
 * backward a reduce-scatter SUM of the dK/dV partials at their owners (NeMo
 * Automodel page "block-diagonal varlen CP for packed sequences", Design
 * overview, exchange.py). dq fp32 [B, nchunks, L, H, d] is overwritten. dk, dv fp32
 * key-like tensors receive each K/V buffer's gradient: in BD_KV_GATHER mode
 * the contributions of all the plan's chunks of a sequence are summed into
 * that sequence's buffer (the reduce-scatter SUM done in place); in
 * BD_KV_WINDOW mode each window buffer receives its own chunk's partial (sum
 * the partials at their owners with bd_owner_sum). accumulate_dkv = 1 adds
 * into dk/dv instead of overwriting (summing successive single-chunk calls).
 * workspace: device memory of bd_attn_bwd_workspace bytes, 256-byte aligned. */
BD_API int32_t bd_attn_bwd(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                    const bd_tensor* k, const bd_tensor* v, const bd_tensor* out,
                    const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq,
                    bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Flags of bd_attn_bwd_ex / bd_attn_bwd_main_ex. */
typedef enum {
  /* dk, dv are owner-row tensors fp32 [B, 1, S', Hkv, d] (S' >= S) instead of
   * key-like ones: every chunk's contribution to key row r of sequence b is
   * summed, deterministically, into dk[b, 0, r] -- the reduce-scatter SUM of
   * the fused all-gather, or the index_add of the needed-only exchange, done in
   * the kernel (NeMo Automodel page "block-diagonal varlen CP for packed
   * sequences", Design overview, exchange.py). Rows at or past s_valid get
   * zeros (with accumulate_dkv = 0). Needs a BD_KV_WINDOW plan over every chunk
   * 0..cp-1 in order with L a multiple of 128 (else BD_ERR_UNSUPPORTED, before
   * any launch); k, v are its window buffers. Equal, up to rounding order, to
   * bd_attn_bwd followed by bd_owner_sum_ex. */
  BD_BWD_OWNER_ROWS = 1,
  /* dq is already zero (bd_attn_fwd_ex cleared it): the statistics step skips
   * clearing it. Ignored by bd_attn_bwd_main_ex. */
  BD_BWD_DQ_ZEROED = 2
} bd_bwd_flags;

/* bd_attn_bwd_ex -- bd_attn_bwd with flags (bd_bwd_flags, OR-ed). Every
 * argument of both steps is checked before the first launch. Unknown flag bits
 * give BD_ERR_ARG. */
BD_API int32_t bd_attn_bwd_ex(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                       const bd_tensor* k, const bd_tensor* v, const bd_tensor* out,
                       const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq,
                       bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv, int32_t flags,
                       void* workspace, size_t workspace_bytes, void* stream);

/* bd_attn_bwd_pre -- the first step of bd_attn_bwd on its own: per row and
 * head D = <dout, out> (fp32) and the LSE in log2 units, written into
 * `workspace`; zeroes dq. out and dout are read by TMA: their base and strides
 * must be 16-byte aligned (else BD_ERR_ALIGN before any launch). */
BD_API int32_t bd_attn_bwd_pre(const void* plan_host, const void* plan_dev, const bd_tensor* out,
                        const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq, void* workspace,
                        size_t workspace_bytes, void* stream);

/* bd_attn_bwd_pre_ex -- bd_attn_bwd_pre with clear_dq = 0 leaving dq as it is:
 * for callers that zero the fp32 dq accumulator themselves, e.g. on another
 * stream while the forward runs (dq must be zero before bd_attn_bwd_main). */
BD_API int32_t bd_attn_bwd_pre_ex(const void* plan_host, const void* plan_dev, const bd_tensor* out,
                           const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq, void* workspace,
                           size_t workspace_bytes, int32_t clear_dq, void* stream);

/* bd_attn_bwd_main -- the second step of bd_attn_bwd on its own: dq (added
 * into what bd_attn_bwd_pre zeroed), dk and dv from the workspace that
 * bd_attn_bwd_pre filled for the same plan and tensors. */
BD_API int32_t bd_attn_bwd_main(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                         const bd_tensor* k, const bd_tensor* v, const bd_tensor* dout, bd_tensor* dq,
                         bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv, void* workspace,
                         size_t workspace_bytes, void* stream);

/* bd_attn_bwd_main_ex -- bd_attn_bwd_main with flags: BD_BWD_OWNER_ROWS sums
 * dk / dv at their owner rows (see bd_bwd_flags). */
BD_API int32_t bd_attn_bwd_main_ex(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                            const bd_tensor* k, const bd_tensor* v, const bd_tensor* dout, bd_tensor* dq,
                            bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv, int32_t flags,
                            void* workspace, size_t workspace_bytes, void* stream);

/* bd_owner_sum -- add the BD_KV_WINDOW partials dk_win/dv_win (key-like fp32,
 * Ck = nchunks) of every chunk of the plan into owner-row tensors dk/dv
 * (fp32 [B, 1, S, Hkv, d]): dk[b, kv_start_c + r] += dk_win[b, c, r] for the
 * window rows r < kv_end_c - kv_start_c. The single-GPU form of the
 * needed-only exchange's index_add / reduce-scatter SUM backward
 * (Design overview, exchange.py). Deterministic: chunks are added in order. */
BD_API int32_t bd_owner_sum(const void* plan_host, const void* plan_dev, const bd_tensor* dk_win,
                     const bd_tensor* dv_win, bd_tensor* dk, bd_tensor* dv, void* stream);

/* bd_owner_sum_ex -- bd_owner_sum with accumulate = 0 storing the sum instead
 * of adding it: every owner row of dk/dv is written (rows no window covers,
 * i.e. padding, get zeros), so they need no clearing and are not read.
 * accumulate = 1 is bd_owner_sum. */
BD_API int32_t bd_owner_sum_ex(const void* plan_host, const void* plan_dev, const bd_tensor* dk_win,
                        const bd_tensor* dv_win, bd_tensor* dk, bd_tensor* dv, int32_t accumulate,
                        void* stream);

/* bd_attn_bwd_noalloc -- bd_attn_bwd for callers that cannot allocate device
 * memory (no allocator is available to them, or a memory cap forbids one
 * more allocation). The NeMo Automodel page has no counterpart: it is an
 * addition of this library. The workspace comes from a fixed 16 MiB array in device global
 * memory declared by the library (held on every GPU that loads it until exit);
 * nothing is allocated. Plans needing more workspace than
 * bd_attn_bwd_noalloc_capacity() return BD_ERR_CAPACITY before any launch.
 * All calls on a device share the array: calls that may overlap on the GPU
 * race and must be ordered by the caller. The first call on a device looks up
 * the array's address; make it before any stream capture. That address is kept
 * until the process exits: resetting the device (cudaDeviceReset) between calls
 * is not supported. Arguments and
 * results are those of bd_attn_bwd without the workspace. */
BD_API int32_t bd_attn_bwd_noalloc(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                            const bd_tensor* k, const bd_tensor* v, const bd_tensor* out,
                            const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq, bd_tensor* dk,
                            bd_tensor* dv, int32_t accumulate_dkv, void* stream);

/* Bytes of workspace bd_attn_bwd_noalloc can serve. */
BD_API size_t bd_attn_bwd_noalloc_capacity(void);

/* Reads the failure status kernels recorded in the device plan (waits for the
 * stream). BD_OK, or BD_ERR_DEVICE_TIMEOUT if a kernel gave up waiting.
 * reset != 0 clears the status afterwards. */
BD_API int32_t bd_check_status(const void* plan_dev, int32_t reset, void* stream);

/* bd_selftest_bounded_wait -- failure-detection self test: launches a one-warp
 * kernel that waits, with the same bounded wait every kernel of the library
 * uses, on an mbarrier nothing arrives at; after limit_us microseconds
 * (1..1e6) the wait gives up and the kernel records BD_ERR_DEVICE_TIMEOUT in
 * the plan's status word, which bd_check_status then reports. Nothing faults
 * and the context stays usable. */
BD_API int32_t bd_selftest_bounded_wait(const void* plan_dev, uint32_t limit_us, void* stream);

/* Message for the calling thread's last non-OK status ("" if none). */
BD_API const char* bd_last_error(void);

/* Library version, e.g. 100 for 0.1.0. */
BD_API int32_t bd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BD_ATTN_H */

/*
 * fa.h -- C ABI of the exact-attention library for GB300 (sm_103a), libfa.so.
 *
 * Exact softmax attention O = softmax(scale * Q K^T [+ causal mask]) V computed
 * tile by tile with an online softmax, so the n x n score and probability
 * matrices never reach device memory.
 *
 * Sources for what each call computes:
 *  - "13.14 FlashAttention: IO-aware exact attention" (textbookofai.com),
 *    sections "Tile decomposition" and "Online softmax": the tiled one-pass
 *    algorithm and its exactness; "Backpropagation uses the same trick": the
 *    backward recomputes tiles instead of storing P.
 *  - "efficient-attention/flash-2-3" (zerotofrontier.app), sections
 *    "Fewer non-matmul FLOPs" (unnormalised output, one division at the end,
 *    lse = m + log l kept for the backward, e^(s - lse) recomputed),
 *    "Parallelism over the sequence" (grid over query blocks x batch*heads;
 *    backward over key blocks with dQ added atomically), "Decoding needs a
 *    different split" (split-KV partials and the log-sum-exp merge),
 *    "Variable-length batches without padding" (packed rows + cu_seqlens),
 *    "Using it, the real way" (flash-attn's (batch, T, heads, d_k) layout).
 *
 * Conventions shared by every call
 *  - Element type: bf16 for Q, K, V, O, dO, dQ, dK, dV; fp32 for lse.
 *  - Dense layout [B, N, H, d] contiguous (d fastest); packed layout
 *    [total, H, d]; lse [B, H, N] dense, [H, total] packed, [B, H] decode.
 *  - lse is the natural log of sum_j exp(scale * q . k_j) (scale included).
 *  - causal: key j is visible to query i iff j <= i (queries and keys have
 *    the same length in every causal call, where the top-left and
 *    bottom-right alignments coincide).
 *  - Supported head dims: d in {64, 128}.
 *  - Ownership: the caller allocates and owns every buffer (device memory);
 *    the library allocates nothing.  Calls that need scratch memory take a
 *    caller-provided workspace sized by the matching *_workspace_bytes().
 *  - Asynchrony: every call only enqueues work on `stream` and returns.
 *  - Errors: arguments are validated on the host before any launch; on an
 *    error nothing is launched and no output is touched.  Device pointers
 *    must be 16-byte aligned (FA_ERR_MISALIGNED otherwise).  A launch failure
 *    gives FA_ERR_LAUNCH.  Every wait inside the kernels is bounded; a wait
 *    that runs out records a code that fa_device_error() returns
 *    (FA_ERR_TIMEOUT) instead of hanging the GPU.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same handle as cudaStream_t; NULL = legacy default stream */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* a size, count or scale out of range, a null pointer */
  FA_ERR_UNSUPPORTED = 2, /* head dim not in {64, 128}, device not sm_103 */
  FA_ERR_MISALIGNED = 3,  /* a device pointer not 16-byte aligned */
  FA_ERR_LAUNCH = 4,      /* the CUDA runtime refused a launch */
  FA_ERR_TIMEOUT = 5,     /* a bounded wait inside a kernel ran out */
  FA_ERR_SCRATCH_LIMIT = 6, /* fa_bwd_noalloc: the problem needs more than its built-in scratch */
  FA_ERR_OUT_OF_PAGES = 7   /* page pool: no free page (or sequence slot) for the request; nothing changed */
} fa_status;

/* Human-readable name of a status code (static storage). */
const char* fa_status_string(fa_status s);

/*
 * Forward pass, dense batch.  ("Tile decomposition", "Online softmax";
 * FlashAttention-2 "Fewer non-matmul FLOPs".)
 *   q, k, v : [B, N, H, d] bf16, device, read only
 *   o       : [B, N, H, d] bf16, device, written
 *   lse     : [B, H, N] fp32, device, written (natural log, scale included)
 *   causal  : 0 or 1
 *   scale   : multiplies Q K^T before the softmax (> 0, finite)
 * B, H >= 1 and N >= 0 (N == 0 is a no-op).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 int causal, float scale, fa_stream_t stream);

/*
 * Grouped-query attention forward ("Using it, the real way": fewer key-value
 * heads than query heads, shared in groups).  Query head h attends with K/V
 * head h / (Hq / Hkv).
 *   q, o    : [B, N, Hq, d] bf16;   lse : [B, Hq, N] fp32
 *   k, v    : [B, N, Hkv, d] bf16, Hkv divides Hq
 * Otherwise as fa_fwd (fa_fwd is this call with Hkv = Hq).
 */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                     int d, int causal, float scale, fa_stream_t stream);

/*
 * Scratch bytes fa_bwd needs: an fp32 dQ accumulator [B, N, H, d] and the
 * row sums D_i = sum_k dO_ik O_ik [B, H, N] fp32.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass, dense batch.  (Backpropagation "recomputes the relevant
 * tiles"; FlashAttention-2: weights recomputed as e^(s - lse), parallel over
 * key blocks, dQ added atomically.)
 *   q, k, v, o : [B, N, H, d] bf16 (o from fa_fwd)
 *   lse        : [B, H, N] fp32 from fa_fwd
 *   dout       : [B, N, H, d] bf16, gradient of the loss with respect to O
 *   dq, dk, dv : [B, N, H, d] bf16, written
 *   workspace  : fa_bwd_workspace_bytes(B, H, N, d) bytes, device, 16-byte
 *                aligned; contents on entry do not matter
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, void* workspace, int B, int H, int N, int d, int causal, float scale,
                 fa_stream_t stream);

/*
 * Grouped-query attention backward: dK and dV of each K/V head sum the
 * contributions of every query head in its group.
 *   q, o, dout, dq : [B, N, Hq, d];  k, v, dk, dv : [B, N, Hkv, d];  lse [B, Hq, N]
 *   workspace      : fa_bwd_workspace_bytes(B, Hq, N, d) bytes
 * Otherwise as fa_bwd.
 */
fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, void* workspace, int B, int Hq, int Hkv, int N, int d, int causal,
                     float scale, fa_stream_t stream);

/*
 * Forward pass, packed variable-length batch ("Variable-length batches
 * without padding").  Sequence b owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1
 * and attends only within them; tiles between sequences are never visited.
 *   q, k, v    : [total_tokens, H, d] bf16
 *   o          : [total_tokens, H, d] bf16, written
 *   lse        : [H, total_tokens] fp32, written
 *   cu_seqlens : int32 [num_seqs + 1], DEVICE memory, non-decreasing,
 *                cu_seqlens[0] = 0, cu_seqlens[num_seqs] = total_tokens
 *   max_seqlen : an upper bound of every sequence length.  A sequence longer
 *                than it, or offsets outside the tensors, are reported by
 *                fa_device_error (FA_ERR_INVALID_ARG, code 0x2001) and nothing
 *                is written for that sequence
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                        int num_seqs, int max_seqlen, int total_tokens, int H, int d, int causal, float scale,
                        fa_stream_t stream);

/* Scratch bytes fa_bwd_varlen needs (same two buffers over total_tokens rows). */
size_t fa_bwd_varlen_workspace_bytes(int total_tokens, int H, int d);

/* Backward pass of fa_fwd_varlen; tensors as in fa_bwd in the packed layout.
 * Sequences longer than max_seqlen or outside the tensors are reported as in
 * fa_fwd_varlen, and their dK, dV rows are not written. */
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, const int* cu_seqlens,
                        int num_seqs, int max_seqlen, int total_tokens, int H, int d, int causal, float scale,
                        fa_stream_t stream);

/*
 * Masked attention: causal or sliding-window masks with their own query and
 * key lengths, as used by chunked prefill against a longer cache
 * ("efficient-attention/flash-2-3", section "Using it, the real way":
 * FlashAttention kernels support causal masks, sliding windows
 * and variable lengths natively; PyTorch's is_causal is aligned to the top
 * left and is wrong for chunked prefill, where the bottom-right alignment of
 * the flash-attn package is the one wanted).
 *
 * Mask, bottom-right aligned: query i of a sequence with Nq queries and Nk keys
 * sits at key position i + Nk - Nq and sees the keys j with
 *     i + Nk - Nq - window_left <= j <= i + Nk - Nq + window_right,
 * a bound of -1 leaving its side open.  (-1, -1) is no mask, (-1, 0) causal,
 * (w, 0) causal with a window of w + 1 keys.  Key tiles that no row of a
 * 128-row query tile sees are never loaded ("create_block_mask ... skips
 * them": block-sparse attention).  A query row that sees no key gets O = 0 and
 * lse = -inf.  Nk = 0 is allowed: every row is such a row.
 *   q, o   : [B, Nq, Hq, d] bf16       k, v : [B, Nk, Hkv, d] bf16 (Hkv divides Hq)
 *   lse    : [B, Hq, Nq] fp32, natural log, written
 *   window_left, window_right : >= -1; values past the sequence mean no bound
 * Returns FA_ERR_INVALID_ARG for a bound below -1; otherwise as fa_fwd_gqa.
 */
fa_status fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, int window_left, int window_right, float scale, fa_stream_t stream);

/*
 * fa_fwd_masked on a packed batch: sequence b owns query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1, and the mask aligns the two at the bottom right.
 *   q, o : [total_q, Hq, d];  k, v : [total_k, Hkv, d];  lse : [Hq, total_q]
 *   cu_seqlens_q, cu_seqlens_k : int32 [num_seqs + 1], DEVICE memory, as in
 *                fa_fwd_varlen; offsets outside the tensors are reported by
 *                fa_device_error (FA_ERR_INVALID_ARG) and nothing is written
 *                for that sequence
 *   max_seqlen_q, max_seqlen_k : upper bounds of the sequences' lengths (a
 *                longer sequence is reported like a bad offset)
 */
fa_status fa_fwd_masked_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs, int max_seqlen_q,
                               int max_seqlen_k, int total_q, int total_k, int Hq, int Hkv, int d, int window_left,
                               int window_right, float scale, fa_stream_t stream);

/*
 * Backward pass of fa_fwd_masked (Nq, Nk >= 1).  dK, dV of keys that no query
 * sees are zero; dK, dV sum over the query heads of each K/V head's group.
 *   q, o, dout, dq : [B, Nq, Hq, d];  k, v, dk, dv : [B, Nk, Hkv, d];  lse [B, Hq, Nq]
 *   workspace      : fa_bwd_workspace_bytes(B, Hq, Nq, d) bytes
 */
fa_status fa_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, int window_left, int window_right, float scale, fa_stream_t stream);

/*
 * Backward pass of fa_fwd_masked_varlen (total_q, total_k >= 1); tensors in the
 * packed layout of the forward.
 *   workspace : fa_bwd_varlen_workspace_bytes(total_q, Hq, d) bytes
 */
fa_status fa_bwd_masked_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, void* workspace,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs, int max_seqlen_q,
                               int max_seqlen_k, int total_q, int total_k, int Hq, int Hkv, int d, int window_left,
                               int window_right, float scale, fa_stream_t stream);

/*
 * FP8 forward, step 1: block quantisation to e4m3 ("efficient-attention/
 * flash-2-3", section "FP8, and the outlier problem": one scale per block of
 * Q, K and V; Q and K first multiplied by a Hadamard matrix times a random
 * +-1 diagonal, "incoherent processing", which spreads outliers over all
 * coordinates).  A block is 128 consecutive rows of one (batch, head).
 *   x         : [B, N, H, d] bf16, device
 *   signs     : int8 [d] of -1 / +1, device (required when rotate = 1)
 *   rotate    : 1 = rows become (x H) * signs, H the Sylvester-Hadamard matrix
 *               with entries +-1 (fast transform in fp32); 0 = as they are
 *   codes     : uint8, written: [B, N, H, d] (transpose = 0), or per head
 *               [B, H, d, n_pad] with n_pad = ceil(N / 128) * 128 and the rows
 *               past N zero (transpose = 1, the layout fa_fwd_fp8 takes for V)
 *   scales    : fp32 [B, H, ceil(N / 128)], written: amax / 448 of each block
 *               (0 for an all-zero block); code = e4m3(x / scale), rounded to
 *               nearest even and saturated at +-448
 * d = 64 or 128; x and codes 16-byte aligned, scales 4-byte aligned.
 */
fa_status fa_fp8_quantize(const void* x, const signed char* signs, void* codes, float* scales, int B, int N, int H,
                          int d, int rotate, int transpose, fa_stream_t stream);

/*
 * FP8 forward, step 2: attention on e4m3 operands (d = 128).  Both products
 * run on the tensor cores in e4m3 with fp32 accumulation; P is rounded to
 * e4m3 (after scaling by its key block's V scale over the head's largest V
 * scale) before the P V product.  Scores are dequantised per pair of tiles,
 * s = (q8 . k8) * q_scale * k_scale * scale (/ d when rotated, since
 * H H^T = d I), and the mask is that of fa_fwd_masked.
 *   q_codes  : [B, Nq, Hq, d] uint8 from fa_fp8_quantize (rotate as "rotated")
 *   k_codes  : [B, Nk, Hkv, d] uint8, same rotation and signs as Q
 *   vt_codes : [B, Hkv, d, ceil(Nk / 128) * 128] uint8 (V, transpose = 1, not rotated)
 *   q_scale, k_scale, v_scale : their block scales
 *   o        : [B, Nq, Hq, d] bf16, written;  lse : [B, Hq, Nq] fp32, written
 * Returns FA_ERR_UNSUPPORTED for d != 128; otherwise as fa_fwd_masked.
 */
fa_status fa_fwd_fp8(const void* q_codes, const void* k_codes, const void* vt_codes, const float* q_scale,
                     const float* k_scale, const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                     int Nk, int d, int window_left, int window_right, int rotated, float scale, fa_stream_t stream);

/*
 * Paged KV cache, write side ("efficient-attention/flash-2-3", section "Paged
 * KV caches, a preview of serving"): the cache is a pool of pages of
 * page_size tokens; each sequence's block table maps its logical blocks to
 * pages; a page is taken from the free list only when the sequence's last
 * page fills; sequences that share a prompt share its pages and copy one only
 * when they would write to it.  The pool object is host memory and does no
 * device work; fa_paged_append moves the data; fa_decode_paged reads it.
 * Policies: the free list is a stack (page 0 is taken first, a released page
 * is the next one taken); a new sequence takes the smallest free slot.
 * The functions are not thread-safe on one pool.
 */
typedef struct fa_page_pool fa_page_pool;

/* A pool of num_pages pages for up to max_seqs sequences of up to max_blocks
 * blocks each; NULL for a size below 1 or when host memory runs out. */
fa_page_pool* fa_pool_create(int num_pages, int page_size, int max_seqs, int max_blocks);
void fa_pool_destroy(fa_page_pool* pool);
int fa_pool_free_pages(const fa_page_pool* pool);          /* -1 for NULL */
int fa_pool_refcount(const fa_page_pool* pool, int page);  /* tables holding the page; -1 if invalid */

/* A new, empty sequence in the smallest free slot (*seq); FA_ERR_OUT_OF_PAGES when none is free. */
fa_status fa_pool_add_seq(fa_page_pool* pool, int* seq);
/* A new sequence (*child) sharing every page of parent, e.g. a common prompt. */
fa_status fa_pool_fork(fa_page_pool* pool, int parent, int* child);
/* Drops a sequence; pages no table holds any more return to the free list. */
fa_status fa_pool_release(fa_page_pool* pool, int seq);

/*
 * Reserves the next token of each of n distinct live sequences seqs[0..n-1]
 * (host arrays): page[i], slot[i] receive where the token goes and
 * copy_src[i] the page to copy into page[i] first (-1 for none: only a shared,
 * partly filled last page is copied).  All or nothing: FA_ERR_OUT_OF_PAGES if
 * the free list cannot cover the batch, FA_ERR_INVALID_ARG for a bad or
 * repeated sequence or a full block table, and then nothing changes.
 */
fa_status fa_pool_reserve_append(fa_page_pool* pool, const int* seqs, int n, int* page, int* slot, int* copy_src);

/* Block tables [max_seqs, max_blocks] (unused entries 0) and lengths [max_seqs], host int32. */
fa_status fa_pool_export(const fa_page_pool* pool, int* block_table, int* seq_lens);

/*
 * Device side of n appends: for entry i, copies page copy_src[i] into page[i]
 * when copy_src[i] >= 0, then writes token i into slot slot[i] of page[i].
 *   k_new, v_new     : [n, Hkv, d] bf16, device
 *   k_pages, v_pages : [num_pages, page_size, Hkv, d] bf16, device, updated
 *   page, slot, copy_src : int32 [n], DEVICE memory (from fa_pool_reserve_append)
 * Entries naming a page outside the pool are skipped and reported by
 * fa_device_error (FA_ERR_INVALID_ARG).  d = 64 or 128.
 */
fa_status fa_paged_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages, const int* page,
                          const int* slot, const int* copy_src, int n, int Hkv, int d, int page_size, int num_pages,
                          fa_stream_t stream);

/*
 * Size of the built-in scratch of fa_bwd_noalloc: 32 MiB of device memory,
 * compiled into the library and held by every GPU that loads it until the
 * process exits.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * Backward pass for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a library-interface variant of fa_bwd.
 *
 * Some callers may not call cudaMalloc or any allocating routine: code
 * running inside a host-side memory budget with no allocator of its own, or a
 * runtime that forbids allocation while it issues work.  This call takes the
 * same inputs and outputs as fa_bwd (dense layout, caller-owned buffers) but
 * no workspace: its scratch (the fp32 dQ accumulator and the per-row D and
 * lse arrays, fa_bwd_workspace_bytes(B, H, N, d) bytes) lives in a fixed
 * array inside the library.  It allocates nothing and calls no allocating
 * routine.
 *
 *   Limit: fa_bwd_workspace_bytes(B, H, N, d) <= FA_BWD_NOALLOC_SCRATCH_BYTES
 *          (for d = 128 about 64 K rows of B*H*N, for d = 64 about 125 K);
 *          larger problems return FA_ERR_SCRATCH_LIMIT without launching.
 *   Set-up: every call looks up the scratch array's device address with the
 *          caller's device current (cudaGetSymbolAddress, which allocates
 *          nothing), so a context created anew after cudaDeviceReset gets the
 *          new address.  On a device's first call the lookup also makes the
 *          runtime load the library's kernels there: make that first call
 *          before any stream capture.
 *   Sharing: every call on a device uses the same scratch.  The kernels clear
 *          what must start at zero, but two calls whose work overlaps on the
 *          GPU (different streams, or host threads racing) corrupt each
 *          other's results: order them on one stream or synchronise.
 * Other arguments and errors as fa_bwd.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                         float scale, fa_stream_t stream);

/*
 * Scratch bytes fa_decode_splitkv needs for num_splits partial results:
 * fp32 O_c [B, H, num_splits, d] and lse_c [B, H, num_splits].
 */
size_t fa_decode_workspace_bytes(int B, int H, int d, int num_splits);

/* Number of splits fa_decode_splitkv uses when it is given num_splits = 0. */
int fa_decode_num_splits(int B, int H, int L, int d);

/*
 * Single-token decode with a split KV cache ("Decoding needs a different
 * split"): each chunk of the cache yields a partial (O_c, lse_c), and a
 * second kernel merges them, lse = log sum_c e^lse_c and
 * O = sum_c e^(lse_c - lse) O_c.
 *   q                : [B, 1, H, d] bf16
 *   k_cache, v_cache : [B, L, H, d] bf16
 *   o                : [B, 1, H, d] bf16, written
 *   lse              : [B, H] fp32, written
 *   num_splits       : 0 = choose (fa_decode_num_splits); else 1..L
 *   workspace        : fa_decode_workspace_bytes(B, H, d, splits) bytes
 */
fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B,
                            int H, int L, int d, int num_splits, void* workspace, float scale, fa_stream_t stream);

/*
 * Grouped-query single-token decode: q [B, 1, Hq, d], caches [B, L, Hkv, d]
 * with Hkv dividing Hq and Hq / Hkv <= 32; every K/V row is read once for
 * all the query heads of its group.  Otherwise as fa_decode_splitkv.
 */
fa_status fa_decode_gqa(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                        int Hkv, int L, int d, int num_splits, void* workspace, float scale, fa_stream_t stream);

/*
 * Single-token decode over a paged KV cache ("Paged KV caches, a preview of
 * serving"): the cache is a pool of fixed-size pages anywhere in memory and
 * each sequence's block table maps its logical blocks (keys 0..P-1, P..2P-1,
 * ...) to physical pages.  The kernel gathers one page per block; everything
 * else is the split-KV decode above.  Only the first seq_lens[b] keys of a
 * sequence are read: slots past it in its last page are never touched.
 *   q                : [B, 1, H, d] bf16
 *   k_pages, v_pages : [num_pages, page_size, H, d] bf16
 *   block_table      : int32 [B, max_blocks], DEVICE memory
 *   seq_lens         : int32 [B], DEVICE memory, each in [0, max_seq_len]
 *   page_size        : a multiple of 4 (16 in the pages' example)
 *   max_seq_len      : <= max_blocks * page_size; sizes the splits
 *   num_splits, workspace, o, lse, scale: as fa_decode_splitkv (workspace
 *   sized with fa_decode_workspace_bytes(B, H, d, splits))
 * A table entry outside [0, num_pages) or a length outside [0, max_seq_len]
 * is not dereferenced: the kernel reads page 0 / clamps the length instead and
 * a following fa_device_error() returns FA_ERR_INVALID_ARG.
 */
fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                          const int* seq_lens, void* o, float* lse, int B, int H, int d, int page_size, int num_pages,
                          int max_blocks, int max_seq_len, int num_splits, void* workspace, float scale,
                          fa_stream_t stream);

/*
 * Decode with a sliding window ("efficient-attention/flash-2-3", section
 * "Using it, the real way": FlashAttention kernels support sliding windows):
 * the single query of sequence b sits at key position len - 1 and sees keys
 * len - 1 - window_left .. len - 1 (window_left = -1: all of them, as
 * fa_decode_gqa).  The splits cover the window only, so a long cache costs
 * what its window does.
 *   window_left : >= -1; a window past every key is no window
 *   workspace   : fa_decode_workspace_bytes(B, Hq, d, splits)
 * Otherwise as fa_decode_gqa.
 */
fa_status fa_decode_window(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                           int Hkv, int L, int d, int window_left, int num_splits, void* workspace, float scale,
                           fa_stream_t stream);

/*
 * fa_decode_paged with grouped K/V heads and a sliding window: q [B, 1, Hq, d],
 * k_pages, v_pages [num_pages, page_size, Hkv, d] (Hkv divides Hq, Hq / Hkv <= 32);
 * sequence b sees its keys seq_lens[b] - 1 - window_left .. seq_lens[b] - 1
 * (window_left = -1: all).  Otherwise as fa_decode_paged.
 */
fa_status fa_decode_paged_window(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                                 const int* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d,
                                 int page_size, int num_pages, int max_blocks, int max_seq_len, int window_left,
                                 int num_splits, void* workspace, float scale, fa_stream_t stream);

/*
 * Synchronises the device, then returns FA_OK if no kernel of this library
 * recorded an error since the last call, FA_ERR_TIMEOUT if a bounded wait ran
 * out (code 0x1000 + wait site), FA_ERR_INVALID_ARG if a kernel met a bad
 * device-side argument (0x2000: block-table entry outside the page pool,
 * 0x2001: sequence length out of range).  The recorded code goes to *code
 * when code is not NULL.  Clears the recorded code.
 */
fa_status fa_device_error(unsigned int* code);

/*
 * Failure-detection self-test: launches one warp that waits, through the same
 * bounded-wait helper every kernel uses, on a barrier nothing ever arrives on.
 * The wait gives up after timeout_ms (1 .. 10000) and records
 * FA_DEVERR_SELFTEST_CODE, so a following fa_device_error() returns
 * FA_ERR_TIMEOUT with that code and the context stays usable.  The pages have
 * no counterpart; this checks the library's guard against hung waits.
 */
#define FA_DEVERR_SELFTEST_CODE 0x10FFu
fa_status fa_selftest_wait_timeout(double timeout_ms, fa_stream_t stream);

/*
 * Self-test of the exponentials the forward kernel can use ("efficient-
 * attention/flash-2-3", section "And on Blackwell": part of the exponentials
 * are computed on the FMA units as 2^x = 2^floor(x) * p3(x - floor(x)) with a
 * cubic p3, instead of on the special-function unit).  Evaluates, for each of
 * the n fp32 values x[i] (device), y[i] = (device, written)
 *   which = 0 : the kernel's cubic (inputs below -127 are clamped to -127;
 *               coefficients fitted in fit_exp2_poly.py, relative error
 *               8.6e-5 on [-126, 0])
 *   which = 1 : the special-function unit's ex2.approx.ftz.f32
 *   which = 2 : CUDA's exp2f
 *   which = 3 : the cubic evaluated two values at a time with the packed
 *               f32x2 instructions (the form the forward kernel uses); bit
 *               for bit equal to which = 0
 * x and y 4-byte aligned.  The pages print no error bound; the test compares
 * the cubic with float64 2^x and with exp2f.
 */
fa_status fa_selftest_exp2(const float* x, float* y, int n, int which, fa_stream_t stream);

/*
 * Developer knobs (process-wide; they change speed, not results beyond
 * rounding):
 *   FA_OPT_RESCALE_TAU   : lazy-rescale threshold in log2 units (default 8;
 *                          0 rescales whenever the running maximum grows)
 *   FA_OPT_POLY_EXP      : share of the forward's softmax exponentials
 *                          evaluated with the cubic on the FMA pipe: 0 = none
 *                          (all on the SFU), 4 / 8 / 16 = one column pair in
 *                          4 / 8 / 16 (default 16), 1 = 8 (bf16
 *                          sliding-window kernels: 4 means 8; FP8 kernels:
 *                          4 means 8, and with a window 16 means none);
 *                          other values give FA_ERR_INVALID_ARG
 *   FA_OPT_WAIT_TIMEOUT_MS : limit of every bounded wait (default 2000)
 */
typedef enum { FA_OPT_RESCALE_TAU = 1, FA_OPT_POLY_EXP = 2, FA_OPT_WAIT_TIMEOUT_MS = 3 } fa_option;
fa_status fa_set_option(fa_option opt, double value);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */

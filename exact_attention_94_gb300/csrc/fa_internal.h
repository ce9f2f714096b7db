// Host-side launch interfaces shared between the C-ABI layer and the kernel
// translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

struct FwdParams {
  void* o;                   // bf16 output
  float* lse;                // fp32 log-sum-exp
  const int* cu_seqlens;     // packed query offsets (device) or nullptr for a dense batch
  const int* cu_seqlens_k;   // packed key offsets (device); set exactly when cu_seqlens is
  int H;                     // query heads
  int kv_group;              // query heads per K/V head (grouped-query attention; 1 = one K/V head per query head)
  int bh_total;              // (batch or sequences) * H
  int n_rows;                // rows along the sequence axis of Q and O (Nq, or total query tokens)
  int n_rows_k;              // rows along the sequence axis of K and V (Nk, or total key tokens)
  int seq_len;               // dense: Nq
  int seq_len_k;             // dense: Nk
  int win_left;              // mask (used by the masked kernels): query i sees keys
  int win_right;             //   [i + Nk - Nq - win_left, i + Nk - Nq + win_right]; -1 = unbounded side
  int num_pairs;             // 256-row query chunks (pairs of 128-row tiles) of the longest sequence
  int couple;                // 1: a CTA computes two chunks of a (sequence, head), P-1-u and u
  int num_items;             // packed batch: grid.y enumerates (sequence, chunk or couple) items and x, z
                             //   the query heads; 0: grid over (batch, head) x chunks (or couples)
  int max_len;               // longest query sequence the caller declared (packed: max_seqlen_q)
  int max_len_k;             // longest key sequence the caller declared
  // e4m3 operands only: one scale per 128-row block, [B][H][n_qblk] for Q and
  // [B][Hkv][n_kblk] for K and V (V's codes are stored transposed per head)
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int n_qblk;
  int n_kblk;
  float scale_log2;          // scale * log2(e) (e4m3 with rotated Q, K: also divided by d)
  float tau;                 // lazy-rescale threshold, log2 units
  unsigned* err;             // device error word
  unsigned long long timeout_ns;
};

struct BwdParams {
  const void* o;
  const void* dout;
  const float* lse;          // natural-log lse from the forward
  float* lse2;               // workspace: lse * log2 e, same layout as lse
  float* dsum;               // workspace: D_i = sum_c dO_ic O_ic, same layout as lse
  float* dq_acc;             // workspace: fp32 [B_tensor*H][d/4][n_rows][4]
  void* dq;
  void* dk;
  void* dv;
  const int* cu_seqlens;     // packed query offsets (device) or nullptr
  const int* cu_seqlens_k;   // packed key offsets (device); set exactly when cu_seqlens is
  int B;                     // dense batch, or number of sequences
  int B_tensor;              // leading extent of the tensors: B (dense) or 1 (packed)
  int H;                     // query heads
  int kv_group;              // query heads per K/V head (1 = one K/V head per query head)
  int n_rows;                // rows along the sequence axis of Q, O, dO, dQ
  int n_rows_k;              // rows along the sequence axis of K, V, dK, dV
  int seq_len;               // dense: Nq
  int seq_len_k;             // dense: Nk
  int win_left;              // mask, as in FwdParams
  int win_right;
  int num_kblocks;           // grid.y of the main kernel
  int num_items;             // packed batch: grid.y enumerates (sequence, key block) items and x, z the
                             //   K/V heads; 0: grid over (batch, K/V head) x key blocks
  int max_len;               // longest query / key sequence the caller declared (packed calls)
  int max_len_k;
  float scale;
  float scale_log2;
  unsigned* err;
  unsigned long long timeout_ns;
};

// Encodes a 4-D bf16 tensor map over [B][n_rows][H][D] with a box_rows x 64-column
// box and 128-byte swizzle.  Returns false when the driver refuses it.
bool make_tmap_bhnd(CUtensorMap* m, const void* ptr, int D, int n_rows, int H, int B, int box_rows = 128);

// Mask kinds the kernels are specialised for: none; a right bound only
// (causal-like, every row's keys start at 0); any other window.
enum MaskKind { kMaskNone = 0, kMaskRight = 1, kMaskWindow = 2 };
inline int mask_kind(int win_left, int win_right) {
  return win_left >= 0 ? kMaskWindow : (win_right >= 0 ? kMaskRight : kMaskNone);
}

// poly: one column pair in `poly` of the softmax exponentials on the FMA-pipe
// cubic (0 = all on the SFU; 4, 8 or 16; masks with a left bound: 0 or 8).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                       int D, int mask, int poly, int grid_x, cudaStream_t stream);

// Forward on e4m3 operands (d = 128): tq, tk over codes [B][N][H][d] (uint8),
// tv over V's codes transposed [B][Hkv][d][n_pad].
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const FwdParams& p,
                           int mask, int poly, int grid_x, cudaStream_t stream);

// Block quantisation to e4m3 (d = 64 or 128): x [B][N][H][d] bf16 -> codes and
// one fp32 scale per 128-row block [B][H][ceil(N/128)].  rotate: multiply each
// row by the Hadamard matrix (fast transform) and then by signs[d] (+-1).
// transpose: codes laid out [B][H][d][n_pad] (n_pad = blocks * 128, zero-filled).
cudaError_t launch_fp8_quantize(const void* x, const int8_t* signs, uint8_t* codes, float* scales, int B, int N,
                                int H, int d, bool rotate, bool transpose, cudaStream_t stream);

// 4-D uint8 tensor map: extents dims[0..3] (dims[0] innermost, contiguous),
// byte strides of dims 1..3, a 128 x box_y box, 128-byte swizzle.
bool make_tmap_u8(CUtensorMap* m, const void* ptr, const uint64_t dims[4], const uint64_t strides[3], int box_y);

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int D, int mask, cudaStream_t stream);

// Keys visible to query row i of a sequence with nq queries and nk keys:
// [key_lo, key_hi).  Bottom-right aligned: query i sits at key position
// i + nk - nq; win_left / win_right < 0 leave that side unbounded.  Causal is
// win_left = -1, win_right = 0.
__host__ __device__ __forceinline__ int mask_key_lo(int i, int nq, int nk, int win_left) {
  if (win_left < 0) return 0;
  const long long lo = (long long)i + nk - nq - win_left;
  return lo < 0 ? 0 : (lo > nk ? nk : (int)lo);
}
__host__ __device__ __forceinline__ int mask_key_hi(int i, int nq, int nk, int win_right) {
  if (win_right < 0) return nk;
  const long long hi = (long long)i + nk - nq + win_right + 1;
  return hi < 0 ? 0 : (hi > nk ? nk : (int)hi);
}

struct DecodeParams {
  const void* q;             // [B, 1, H, d] bf16
  const void* k;             // [B, L, H, d] bf16
  const void* v;
  float* part_o;             // [B, H, num_splits, d] fp32: each chunk's normalised output
  float* part_lse;           // [B, H, num_splits] fp32: each chunk's log2 softmax mass
  int B;
  int H;                     // query heads
  int Hkv;                   // K/V heads (grouped-query attention: H = Hkv * kv_group)
  int kv_group;
  int L;
  int G;                     // K/V heads per CTA (divides Hkv; G * kv_group <= 32 query heads)
  int chunk;                 // keys per split
  int num_splits;
  int stages;                // shared-memory ring depth
  int win_left;              // sliding window: only keys >= len - 1 - win_left are seen (-1: all)
  // paged cache (block_table == nullptr: contiguous [B, L, H, d] cache)
  const int* block_table;    // [B, max_blocks] physical page of each logical block of page_size keys
  const int* seq_lens;       // [B] keys of each sequence (<= L)
  int page_size;
  int max_blocks;
  int num_pages;
  float scale_log2;
  unsigned* err;
  unsigned long long timeout_ns;
};

// Paged cache appends: n CTAs, one per token (see fa_paged_append in fa.h).
cudaError_t launch_paged_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages, const int* page,
                                const int* slot, const int* copy_src, int n, int Hkv, int d, int page_size,
                                int num_pages, unsigned* err, cudaStream_t stream);

int decode_stages(int G, int D);
size_t decode_smem_bytes(int G, int D);
cudaError_t launch_decode(const DecodeParams& p, int D, void* o, float* lse, cudaStream_t stream);

}  // namespace fa

// Backward kernels: gradients of exact attention by recomputation.
//
// Method ("13.14 FlashAttention: IO-aware exact attention", "Backpropagation
// uses the same trick": tiles of P are recomputed instead of stored;
// FlashAttention-2 in "efficient-attention/flash-2-3": each weight is
// recomputed as e^(s - lse), the backward is parallel over key blocks, and
// many blocks add into the same dQ_i with atomic additions):
//
//   pre:   D_i = sum_c dO_ic O_ic;  lse2_i = lse_i * log2 e;  dQacc = 0
//   main:  one CTA per 128-key block K_j, V_j; for every 128-row query step i
//          that sees a key of the block (all of them without a mask):
//            S^T  = K_j Q_i^T                 (tcgen05, TMEM)
//            dP^T = V_j dO_i^T                (tcgen05, TMEM)
//            P^T  = 2^(S^T scale log2 e - lse2)       (bf16, back into TMEM)
//            dS^T = scale * P^T * (dP^T - D)          (bf16, shared memory)
//            dV_j += P^T dO_i;  dK_j += dS^T Q_i      (tcgen05, TMEM accumulators)
//            dQ_i  = dS K_j  -> added into dQacc with vector atomics
//   post:  dQ = bf16(dQacc)
//
// The fp32 dQ accumulator is laid out per d (see acc_f4_index) so that a
// warp's atomics always cover contiguous bytes.  The main kernel is described
// above fa_bwd_main_ov_kernel.
#include "fa_internal.h"
#include "ptx.cuh"

#include <climits>
#include <cmath>

namespace fa {

namespace {

constexpr int kBwdHeadGroup = 8;

}  // namespace

// ---------------------------------------------------------------- pre / post

// The fp32 dQ accumulator is kept in one of two layouts (as float4 groups):
//   d = 64 : [B*H][d/4][rows][4]  (the query-row threads of a warp add 512 contiguous bytes)
//   d = 128: [B*H][rows][d]       (the d-row threads of a warp add 128 contiguous bytes)
template <int D>
__host__ __device__ __forceinline__ size_t acc_f4_index(size_t bh, int n_rows, int row, int c4) {
  if constexpr (D == 128)
    return (bh * n_rows + row) * (D / 4) + c4;
  else
    return (bh * (D / 4) + c4) * n_rows + row;
}

// The prologue and epilogue kernels work on tiles of 64 rows of one (batch,
// head): O and dO rows (b, n, h) of d elements, 16 bytes per thread and four
// rows of loads in flight, the index arithmetic done once per CTA.
constexpr int kRowTile = 64;

__device__ __forceinline__ void row_tile_of(int H, int n_rows, long long& bh, int& n0) {
  const int n_tiles = (n_rows + kRowTile - 1) / kRowTile;
  bh = (long long)blockIdx.x / n_tiles;
  n0 = (int)((long long)blockIdx.x - bh * n_tiles) * kRowTile;
}

__device__ __forceinline__ float dot_bf16x8(uint4 a, uint4 b) {
  const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ua[i]));
    const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ub[i]));
    acc = fmaf(fa.x, fb.x, fmaf(fa.y, fb.y, acc));
  }
  return acc;
}

// Per row (b, h, n): D = sum_c dO * O and lse2 = lse * log2 e; the tile's rows
// of the dQ accumulator are zeroed.  Tensors [Bt][rows][H][d].
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        const float* __restrict__ lse, float* __restrict__ dsum,
                                                        float* __restrict__ lse2, float* __restrict__ dq_acc,
                                                        int H, int n_rows) {
  constexpr int TPR = D / 8;              // threads per row, 8 columns each
  constexpr int RPP = 256 / TPR;          // rows per pass
  constexpr int PASSES = kRowTile / RPP;
  long long bh;
  int n0;
  row_tile_of(H, n_rows, bh, n0);
  const long long bt = bh / H;
  const int h = (int)(bh - bt * H);
  const int c8 = (int)threadIdx.x % TPR, rl = (int)threadIdx.x / TPR;
  uint4 a[PASSES], b[PASSES];
#pragma unroll
  for (int k = 0; k < PASSES; ++k) {
    const int n = n0 + rl + k * RPP;
    a[k] = b[k] = make_uint4(0u, 0u, 0u, 0u);
    if (n < n_rows) {
      const size_t off = (((size_t)bt * n_rows + n) * H + h) * D + c8 * 8;
      a[k] = *reinterpret_cast<const uint4*>(o + off);
      b[k] = *reinterpret_cast<const uint4*>(dout + off);
    }
  }
#pragma unroll
  for (int k = 0; k < PASSES; ++k) {
    float acc = dot_bf16x8(a[k], b[k]);
#pragma unroll
    for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    const int n = n0 + rl + k * RPP;
    if (c8 == 0 && n < n_rows) {
      const size_t ri = (size_t)bh * n_rows + n;
      dsum[ri] = acc;
      lse2[ri] = lse[ri] * 1.4426950408889634f;
    }
  }
  // zero the tile's accumulator rows: 64 rows x d/4 groups of 4 floats
  float4* acc4 = reinterpret_cast<float4*>(dq_acc);
#pragma unroll
  for (int k = 0; k < kRowTile * (D / 4) / 256; ++k) {
    const int i = (int)threadIdx.x + 256 * k;
    // d = 128: row-major tile, a row's 32 groups contiguous; d = 64: 16 planes of 64 rows
    const int row = D == 128 ? i / (D / 4) : i % kRowTile;
    const int c4 = D == 128 ? i % (D / 4) : i / kRowTile;
    if (n0 + row < n_rows) acc4[acc_f4_index<D>((size_t)bh, n_rows, n0 + row, c4)] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// dq[bt][n][h][c] = bf16(dQ accumulator).
//   d = 128: 8 columns per thread; a row's 16 threads read 512 contiguous
//            accumulator bytes and write the row's 256 bytes.
//   d = 64 : 16 columns per thread; the 32 threads of a warp take 32
//            consecutive rows of one 16-column group (four planes of the
//            [B*H][d/4][rows][4] layout, 512 contiguous bytes each) and write
//            32 bytes (one L2 sector) of their row each.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_post_kernel(const float* __restrict__ dq_acc,
                                                         __nv_bfloat16* __restrict__ dq, int H, int n_rows) {
  long long bh;
  int n0;
  row_tile_of(H, n_rows, bh, n0);
  const long long bt = bh / H;
  const int h = (int)(bh - bt * H);
  const float4* acc4 = reinterpret_cast<const float4*>(dq_acc);
  if constexpr (D == 128) {
    constexpr int TPR = D / 8;
    constexpr int RPP = 256 / TPR;
    constexpr int PASSES = kRowTile / RPP;
    const int c8 = (int)threadIdx.x % TPR, rl = (int)threadIdx.x / TPR;
    float4 v0[PASSES], v1[PASSES];
#pragma unroll
    for (int k = 0; k < PASSES; ++k) {
      const int n = n0 + rl + k * RPP;
      v0[k] = v1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n < n_rows) {
        v0[k] = acc4[acc_f4_index<D>((size_t)bh, n_rows, n, 2 * c8)];
        v1[k] = acc4[acc_f4_index<D>((size_t)bh, n_rows, n, 2 * c8 + 1)];
      }
    }
#pragma unroll
    for (int k = 0; k < PASSES; ++k) {
      const int n = n0 + rl + k * RPP;
      if (n < n_rows) {
        const uint4 out = make_uint4(pack_bf16x2(v0[k].x, v0[k].y), pack_bf16x2(v0[k].z, v0[k].w),
                                     pack_bf16x2(v1[k].x, v1[k].y), pack_bf16x2(v1[k].z, v1[k].w));
        *reinterpret_cast<uint4*>(dq + (((size_t)bt * n_rows + n) * H + h) * D + c8 * 8) = out;
      }
    }
  } else {
    const int warp = (int)threadIdx.x >> 5;
    const int c16 = warp & 3;                                  // columns 16 * c16 .. + 15
    const int n = n0 + (warp >> 2) * 32 + (int)(threadIdx.x & 31);  // 8 warps: 4 groups x 2 x 32 rows
    if (n < n_rows) {
      uint32_t pk[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 a = acc4[acc_f4_index<D>((size_t)bh, n_rows, n, 4 * c16 + j)];
        pk[2 * j] = pack_bf16x2(a.x, a.y);
        pk[2 * j + 1] = pack_bf16x2(a.z, a.w);
      }
      __nv_bfloat16* dst = dq + (((size_t)bt * n_rows + n) * H + h) * D + c16 * 16;
      if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
        st_global_v8(dst, pk);
      } else {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
  }
}

// ---------------------------------------------------------------- work items and masks

// A backward CTA owns key block [k0, k0 + 128) of one (sequence, K/V head) and
// walks the query rows [q_lo, q_hi) that see at least one of its keys.  With
// the bottom-right mask, query i sees keys [i + off - win_left, i + off +
// win_right], off = kv_len - seq_len, so those rows are
//   q_lo = k0 - off - win_right,  q_hi = k0 + 127 - off + win_left + 1
// (clamped to [0, seq_len); an unbounded side leaves the full range).
struct BwdItem {
  int seq_start, seq_len;  // query rows of the sequence
  int kv_start, kv_len;    // key rows of the sequence
  int b_coord;             // batch coordinate of the tensors (0 when packed)
  int off;                 // kv_len - seq_len
  int q_lo, q_hi;
  bool bad;                // packed offsets outside the tensors, or longer than the stated maxima
};

template <int MASK>
__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int b, int k0) {
  BwdItem it{0, p.seq_len, 0, p.seq_len_k, b, 0, 0, 0, false};
  if (p.cu_seqlens != nullptr) {
    it.seq_start = p.cu_seqlens[b];
    it.seq_len = p.cu_seqlens[b + 1] - it.seq_start;
    it.kv_start = p.cu_seqlens_k[b];
    it.kv_len = p.cu_seqlens_k[b + 1] - it.kv_start;
    it.b_coord = 0;
    it.bad = it.seq_start < 0 || it.seq_len < 0 || it.seq_start > p.n_rows - it.seq_len || it.kv_start < 0 ||
             it.kv_len < 0 || it.kv_start > p.n_rows_k - it.kv_len || it.seq_len > p.max_len ||
             it.kv_len > p.max_len_k;  // a sequence longer than the stated maximum would lose rows
  }
  it.off = it.kv_len - it.seq_len;
  it.q_lo = 0;
  it.q_hi = it.seq_len;
  if (MASK != kMaskNone && p.win_right >= 0) it.q_lo = max(0, k0 - it.off - p.win_right);
  if (MASK == kMaskWindow) it.q_hi = min(it.seq_len, k0 + 128 - it.off + p.win_left);
  return it;
}

// Query q is hidden from key kg iff q < mask_a(kg) or q > mask_b(kg).
template <int MASK>
__device__ __forceinline__ int mask_a(const BwdParams& p, const BwdItem& it, int kg) {
  return (MASK != kMaskNone && p.win_right >= 0) ? kg - it.off - p.win_right : INT_MIN;
}
template <int MASK>
__device__ __forceinline__ int mask_b(const BwdParams& p, const BwdItem& it, int kg) {
  return MASK == kMaskWindow ? kg - it.off + p.win_left : INT_MAX;
}
// Whether some (key, query) pair of keys [k0, k0 + 128) x queries [qs, qs + nq) is hidden.
template <int MASK>
__device__ __forceinline__ bool mask_needed(const BwdParams& p, const BwdItem& it, int k0, int qs, int nq) {
  if (MASK == kMaskNone) return false;
  return (p.win_right >= 0 && qs < k0 + 127 - it.off - p.win_right) ||
         (MASK == kMaskWindow && qs + nq - 1 > k0 - it.off + p.win_left);
}

// No query sees the key block: its dK and dV rows are zero.
template <int D>
__device__ void bwd_zero_dkdv(const BwdParams& p, const BwdItem& it, int Hkv, int h_kv, int k0) {
  const int nk = min(128, it.kv_len - k0);
  for (int idx = (int)threadIdx.x; idx < nk * (D / 8); idx += (int)blockDim.x) {
    const int r = idx / (D / 8), c = idx % (D / 8);
    const size_t grow = ((size_t)it.b_coord * p.n_rows_k + it.kv_start + k0 + r) * Hkv + h_kv;
    if (!FA_INB(grow * D + c * 8, grow * D + c * 8 + 7, (long long)p.B_tensor * p.n_rows_k * Hkv * D, p.err, 17))
      continue;
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk) + grow * D)[c] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dv) + grow * D)[c] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------- main

// ---------------------------------------------------------------- main, overlapped
//
// Steps of 128 queries, so S^T and dP^T are M = 128, N = 128 tcgen05.mma
// (a measured 8192 FLOP/clk/SM; N = 64 reaches only two thirds of that).
// Two warpgroups recompute P and dS: group g owns the step's queries
// [64g, 64g+64) and hands them to the tensor pipe in two quarters of 32, P
// first (for dV) and dS after (for dK), so the products of one quarter run
// while the next is being recomputed.
// d = 128: dQ is produced transposed, dQ^T = K^T dS^T (M = d), into the dP^T
// columns once both groups have read them, and drained while S^T of the next
// step runs.  d = 64: dQ = dS K (M = 128 queries, N = 64) has columns of its own.
//   TMEM: S^T/P^T [0,128), dP^T (d = 128: and dQ^T) [128,256), dV [256,256+d),
//   dK [256+d,256+2d), dQ (d = 64) [384,448).
//   P^T of query q sits at column 64*(q/64) + (q%64)/2: over the recomputing
//   group's own, already-read S^T columns.
//   Shared: K_j, V_j (128 x d each); stages of Q_i, dO_i (two for d = 128,
//           three for d = 64); dS^T 128 keys x 128 queries (two 64-query chunks).
// Warps: 0-3 and 12-15 drain dQ (d = 128: query columns 0-63 and 64-127 of
// dQ^T; d = 64: d columns 0-31 and 32-63 of dQ), 4-11 recompute P and dS,
// 16 issues TMA loads and 17 owns TMEM and issues the MMAs (each warp runs its
// loop with all lanes; an elect.sync lane issues each copy or product).
constexpr int kBwd128Threads = 576;
constexpr int kWarpProducer = 16;
constexpr int kWarpMma = 17;

template <int D>
struct Bwd128Layout {
  static constexpr uint32_t kTile = 128u * D * 2u;     // 128 rows x d
  static constexpr uint32_t kChunk = 128u * 128u;      // 128 rows x 64 columns
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kTile;
  static constexpr uint32_t kStage0 = 2 * kTile;
  static constexpr uint32_t kStageBytes = 2 * kTile;  // Q_i then dO_i
  static constexpr uint32_t kDS = kStage0 + kStages * kStageBytes;
  static constexpr uint32_t kBar = kDS + 2 * kChunk;
  static constexpr uint32_t kBytes = kBar + 256 + 1024 + 1024;  // barriers, lse2/D rows, alignment slack
};

template <int D, int MASK>
__global__ void __launch_bounds__(kBwd128Threads, 1)
    fa_bwd_main_ov_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const BwdParams p) {
  using L = Bwd128Layout<D>;
  constexpr int CH = D / 64;  // 128-byte swizzle columns per row
  constexpr int NST = L::kStages;
  constexpr uint32_t CHUNK = L::kChunk;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);

  const int warp = warp_id();
  const int lane = lane_id();

  // one CTA per (batch, K/V head, key block); with grouped-query attention it
  // walks the query blocks of every query head that shares this K/V head
  // Packed batches with an item list: y enumerates the (sequence, key block)
  // items that exist and x, z the K/V heads.
  const int Hkv = p.H / p.kv_group;
  int b, h_kv, jb;
  if (p.num_items > 0) {
    h_kv = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (h_kv >= Hkv) return;
    int units, total;
    const bool found = varlen_item(p.cu_seqlens_k, p.B, 128, (int)blockIdx.y, b, jb, units, total);
    if (blockIdx.y == gridDim.y - 1 && h_kv == 0 && total > (int)gridDim.y && threadIdx.x == 0 && p.err != nullptr)
      atomicCAS(p.err, 0u, FA_DEVERR_BAD_SEQLEN);  // more items than the grid: the offsets are not as declared
    if (!found) return;
  } else {
    const int bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (bh >= p.B * Hkv) return;
    b = bh / Hkv;
    h_kv = bh % Hkv;
    jb = (int)blockIdx.y;
  }
  const int k0 = jb * 128;
  const BwdItem it = bwd_item<MASK>(p, b, k0);
  if (it.bad) {
    if (threadIdx.x == 0 && p.err != nullptr) atomicCAS(p.err, 0u, FA_DEVERR_BAD_SEQLEN);
    return;
  }
  const int seq_start = it.seq_start, seq_len = it.seq_len, kv_start = it.kv_start, b_coord = it.b_coord;
  if (k0 >= it.kv_len) return;
  const int q_begin = it.q_lo;
  const int n_q = it.q_hi > it.q_lo ? (it.q_hi - it.q_lo + 127) / 128 : 0;  // query blocks per query head
  if (n_q == 0) {  // uniform for the CTA, before any shared state exists
    bwd_zero_dkdv<D>(p, it, Hkv, h_kv, k0);
    return;
  }
  const int n_steps = p.kv_group * n_q;              // step n: query head hq(n), block n % n_q
  auto hq_of = [&](int n) { return h_kv * p.kv_group + n / n_q; };
  auto row_base_of = [&](int hq) { return (size_t)(b_coord * p.H + hq) * p.n_rows + seq_start; };

  enum { KV_FULL = 0, Q_FULL = 1, DO_FULL = Q_FULL + NST, STAGE_EMPTY = DO_FULL + NST, S_FULL = STAGE_EMPTY + NST,
         DP_FULL = S_FULL + 1,
         P_READY = DP_FULL + 1, DS_READY = P_READY + 4,
         DQ_FULL = DS_READY + 4, DQ_EMPTY, DKV_FINAL, DRAIN, NBARS };
  const uint32_t bar0 = base + L::kBar;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + L::kBar + 8 * NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_lse2 = reinterpret_cast<float*>(sbase + L::kBar + 256);  // 128 floats
  float* s_dsum = s_lse2 + 128;                                     // 128 floats

  if (threadIdx.x == 0) {
    mbar_init(BAR(KV_FULL), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(BAR(Q_FULL + s), 1);
      mbar_init(BAR(DO_FULL + s), 1);
      mbar_init(BAR(STAGE_EMPTY + s), 1);
    }
    mbar_init(BAR(S_FULL), 1);
    mbar_init(BAR(DP_FULL), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(BAR(P_READY + i), 128);
      mbar_init(BAR(DS_READY + i), 128);
    }
    mbar_init(BAR(DQ_FULL), 1);
    mbar_init(BAR(DQ_EMPTY), 256);
    mbar_init(BAR(DKV_FINAL), 1);
    mbar_init(BAR(DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx w{abort_flag, p.timeout_ns, p.err};

  const uint32_t sK = base + L::kK, sV = base + L::kV, sDS = base + L::kDS;
  auto stage_q = [&](int st) -> uint32_t { return base + L::kStage0 + (uint32_t)st * L::kStageBytes; };

  if (warp == kWarpProducer) {
    // ============================================================ TMA producer
    // the whole warp runs the loop; one elected lane issues the copies
    {
      if (elect_one()) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        mbar_arrive_expect_tx(BAR(KV_FULL), 2 * L::kTile);
        for (int c = 0; c < CH; ++c) {
          tma_load_4d(sK + c * CHUNK, &tm_k, BAR(KV_FULL), c * 64, kv_start + k0, h_kv, b_coord);
          tma_load_4d(sV + c * CHUNK, &tm_v, BAR(KV_FULL), c * 64, kv_start + k0, h_kv, b_coord);
        }
      }
      bool ok = true;
      for (int n = 0; n < n_steps && ok; ++n) {
        const int st = n % NST;
        const int row = seq_start + q_begin + (n % n_q) * 128;
        const int hq = hq_of(n);
        if (n >= NST &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(BAR(STAGE_EMPTY + st), ((n / NST) - 1) & 1, w, 51))))
          break;
        const uint32_t qa = stage_q(st);
        // Q_i first: S^T of a step is issued while the previous step's products still run
        if (elect_one()) {
          mbar_arrive_expect_tx(BAR(Q_FULL + st), L::kTile);
          for (int c = 0; c < CH; ++c) tma_load_4d(qa + c * CHUNK, &tm_q, BAR(Q_FULL + st), c * 64, row, hq, b_coord);
          mbar_arrive_expect_tx(BAR(DO_FULL + st), L::kTile);
          for (int c = 0; c < CH; ++c)
            tma_load_4d(qa + L::kTile + c * CHUNK, &tm_do, BAR(DO_FULL + st), c * 64, row, hq, b_coord);
        }
      }
      if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ============================================================ MMA issuer
    // the whole warp runs the loop; one elected lane issues each product and commit
    {
      constexpr uint32_t IDESC_SD = idesc_bf16(128, 128, false, false);  // S^T, dP^T: M keys, N queries
      constexpr uint32_t IDESC_KV = idesc_bf16(128, D, false, true);     // dV, dK: M keys, N d
      // d = 128: dQ^T, M d, N queries, both operands MN-major; d = 64: dQ, M queries, N d, both MN-major
      constexpr uint32_t IDESC_DQ = idesc_bf16(128, 128, true, true);
      const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 256 + D, tDQ = tmem + 384;
      // base descriptors; each product only advances the start address
      const uint64_t dK_kmaj = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dV_kmaj = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dK_mn = smem_desc_sw128(sK, CHUNK, 1024);   // K_j^T as MN-major A over d
      const uint64_t dDS_k = smem_desc_sw128(sDS, 16, 1024);     // dS^T as K-major A (rows = keys)
      const uint64_t dDS_mn = smem_desc_sw128(sDS, CHUNK, 1024); // dS^T as MN-major B over queries
      bool ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_FULL), 0, w, 52));
      tc_fence_after();
      // S^T(n) = K_j Q_n^T into columns [0,128)
      auto issue_s = [&](int n) {
        const int st = n % NST;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(Q_FULL + st), (n / NST) & 1, w, 53)))) return;
        tc_fence_after();
        const uint64_t q_k = smem_desc_sw128(stage_q(st), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * CHUNK + (kk % 4) * 32;
          mma_ss_w(tS, desc_add(dK_kmaj, off), desc_add(q_k, off), IDESC_SD, kk > 0);
        }
        mma_commit_w(BAR(S_FULL));
      };
      if (ok) issue_s(0);
      // Per step n the pipe runs dV(n) quarter by quarter with dP(n) after the first half,
      // then S^T(n+1) (its P is recomputed while dK(n), dQ(n) and dP(n+1) run), then dK(n)
      // as the dS quarters arrive, then dQ(n).  Products issued by one thread execute in
      // order, so S^T(n+1) overwrites P^T(n) only after the dV(n) products have read it.
      for (int n = 0; n < n_steps && ok; ++n) {
        const int st = n % NST;
        const uint32_t qa = stage_q(st), da = qa + L::kTile;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(DO_FULL + st), (n / NST) & 1, w, 62)))) break;
        tc_fence_after();
        const uint64_t do_k = smem_desc_sw128(da, 16, 1024);
        const uint64_t q_mn = smem_desc_sw128(qa, CHUNK, 1024), do_mn = smem_desc_sw128(da, CHUNK, 1024);
        // dV += P^T dO_i, one 32-query quarter at a time as the groups hand them over:
        // quarter i = group (i & 1), half (i >> 1); queries qb .. qb+31 with qb = 64*group + 32*half.
#pragma unroll
        for (int r = 0; r < 2 && ok; ++r) {
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int i = 2 * r + g, qb = 64 * g + 32 * r;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(P_READY + i), n & 1, w, 55)))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint32_t acc = (n > 0 || i > 0 || kk > 0) ? 1u : 0u;
              const uint32_t rows = (uint32_t)(qb / 16 + kk) * 2048;  // 16 query rows of dO_i
              mma_ts_w(tDV, tS + 64 * g + 16 * r + 8 * kk, desc_add(do_mn, rows), IDESC_KV, acc);
            }
          }
          if (r == 0 && ok) {
            if (D == 128 && n > 0) {  // the previous dQ^T must have left the dP^T columns
              if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(DQ_EMPTY), (n - 1) & 1, w, 54)))) break;
              tc_fence_after();
            }
            // dP^T = V_j dO_i^T
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * CHUNK + (kk % 4) * 32;
              mma_ss_w(tDP, desc_add(dV_kmaj, off), desc_add(do_k, off), IDESC_SD, kk > 0);
            }
            mma_commit_w(BAR(DP_FULL));
          }
        }
        if (!ok) break;
        if (n + 1 < n_steps) {
          issue_s(n + 1);
          if (!ok) break;
        }
        // dK += dS^T Q_i as the dS quarters arrive
#pragma unroll
        for (int i = 0; i < 4 && ok; ++i) {
          const int r = i >> 1, g = i & 1, qb = 64 * g + 32 * r;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(DS_READY + i), n & 1, w, 56)))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint32_t acc = (n > 0 || i > 0 || kk > 0) ? 1u : 0u;
            const uint32_t rows = (uint32_t)(qb / 16 + kk) * 2048;  // 16 query rows of Q_i
            mma_ss_w(tDK, desc_add(dDS_k, g * CHUNK + (2 * r + kk) * 32), desc_add(q_mn, rows), IDESC_KV, acc);
          }
        }
        if (!ok) break;
        mma_commit_w(BAR(STAGE_EMPTY + st));
        if constexpr (D == 128) {
          // dQ^T = K_j^T dS^T (M = d, N = 128 queries over both dS^T chunks, K = 128 keys) into the dP^T columns
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_w(tDP, desc_add(dK_mn, kk * 2048), desc_add(dDS_mn, kk * 2048), IDESC_DQ, kk > 0);
        } else {
          // dQ = dS K_j (M = 128 queries, N = d, K = 128 keys): A is dS^T read MN-major over the
          // queries, B is K_j read MN-major over d; its own columns, free once the previous one is drained
          if (n > 0) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(DQ_EMPTY), (n - 1) & 1, w, 54)))) break;
            tc_fence_after();
          }
          constexpr uint32_t IDESC_DQ64 = idesc_bf16(128, D, true, true);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_w(tDQ, desc_add(dDS_mn, kk * 2048), desc_add(dK_mn, kk * 2048), IDESC_DQ64, kk > 0);
        }
        mma_commit_w(BAR(DQ_FULL));
      }
      if (ok) mma_commit_w(BAR(DKV_FINAL));
      mma_commit_w(BAR(DRAIN));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(DRAIN), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ============================================================ P and dS (thread = key row)
    const int g = (warp - 4) >> 2;  // group: queries [64g, 64g+64) of each step
    const int kw = warp & 3;
    const int kr = kw * 32 + lane;
    const int kg = k0 + kr;
    const bool row_ok = kg < it.kv_len;
    const int ma = mask_a<MASK>(p, it, kg), mb = mask_b<MASK>(p, it, kg);
    const uint32_t lane_off = (uint32_t)(kw * 32) << 16;
    const int swz = kr & 7;
    float* my_lse2 = s_lse2 + 64 * g;
    float* my_dsum = s_dsum + 64 * g;
    // Thread kr < 64 carries lse2 of query kr of the group's slice, thread
    // kr >= 64 its D, loaded one step ahead.  The load is left raw until it
    // is staged a step later as the FMA addends -lse2 and -scale * D, so its
    // latency hides under a whole step.  Queries past the end: -lse2 = -inf
    // (so P = 0) and D = 0.
    const float* fsrc = kr < 64 ? p.lse2 : p.dsum;
    int f_blk = 0, f_hq = h_kv * p.kv_group;  // query block and head of the next step to fetch
    const int hq_end = f_hq + p.kv_group;
    float f_raw = 0.f;
    bool f_ok = false;
    auto fetch = [&]() {
      const int qg = q_begin + f_blk * 128 + 64 * g + (kr & 63);
      f_ok = f_hq < hq_end && qg < seq_len &&
             FA_INB(row_base_of(f_hq) + qg, row_base_of(f_hq) + qg, (long long)p.B_tensor * p.H * p.n_rows, p.err, 13);
      f_raw = f_ok ? fsrc[row_base_of(f_hq) + qg] : 0.f;
      if (++f_blk == n_q) {
        f_blk = 0;
        ++f_hq;
      }
    };
    fetch();
    bool ok = true;
    int blk = 0;  // query block of step n
    for (int n = 0; n < n_steps; ++n) {
      const int qs = q_begin + blk * 128 + 64 * g;  // first query of the group's slice
      if (++blk == n_q) blk = 0;
      asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
      if (kr < 64)
        my_lse2[kr] = f_ok ? -f_raw : -INFINITY;
      else
        my_dsum[kr - 64] = f_ok ? -p.scale * f_raw : 0.f;
      asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
      fetch();
      // After an abort the warp keeps taking part in the named barriers and does nothing else.
      if (!ok) continue;
      ok = mbar_wait(BAR(S_FULL), n & 1, w, 57);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        continue;
      }
      tc_fence_after();
      const bool masked = mask_needed<MASK>(p, it, k0, qs, 64);
      const bool tail_rows = k0 + 128 > it.kv_len;  // only the last key block has rows past the end
      const float sl2 = p.scale_log2, scale = p.scale;
      const uint64_t sl2x2 = f2_pack(sl2, sl2), scale2 = f2_pack(scale, scale);
      uint8_t* ds_row = sbase + L::kDS + g * CHUNK + kr * 128;
      // ---- P of both quarters (needs S^T only), each handed to the dV products at once.
      // P is kept as the bf16 pairs the dV product reads until dS needs it.
      uint32_t pp[32];
#pragma unroll
      for (int r = 0; r < 2; ++r) {  // quarter: 32 queries
        const uint32_t col = 64u * g + 32u * r;  // S^T columns of the quarter
        uint32_t sr[32];
        tmem_ld16(tmem + lane_off + col, sr);
        tmem_ld16(tmem + lane_off + col + 16, sr + 16);
        tmem_ld_wait();
        const float4* nl4 = reinterpret_cast<const float4*>(my_lse2 + 32 * r);  // -lse2
        // P = 2^(s * scale * log2 e - lse2)
        float pv[32];
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 nl = nl4[e4];
          // packed f32x2 FMAs: the same fused results as the scalar ones
          float y0, y1, y2, y3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * e4 + 0]), __uint_as_float(sr[4 * e4 + 1])), sl2x2,
                           f2_pack(nl.x, nl.y)), y0, y1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * e4 + 2]), __uint_as_float(sr[4 * e4 + 3])), sl2x2,
                           f2_pack(nl.z, nl.w)), y2, y3);
          pv[4 * e4 + 0] = ex2_sfu(y0);
          pv[4 * e4 + 1] = ex2_sfu(y1);
          pv[4 * e4 + 2] = ex2_sfu(y2);
          pv[4 * e4 + 3] = ex2_sfu(y3);
        }
        if (masked || (tail_rows && !row_ok)) {  // masks in a separate, warp-uniform pass
          const int q32 = qs + 32 * r;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!row_ok || (masked && (q32 + e < ma || q32 + e > mb))) pv[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) pp[16 * r + e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
        // P^T over this group's already-read S^T columns: query q at column 64*(q/64) + (q%64)/2
        tmem_st8(tmem + lane_off + 64u * g + 16u * r, pp + 16 * r);
        tmem_st8(tmem + lane_off + 64u * g + 16u * r + 8u, pp + 16 * r + 8);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(P_READY + 2 * r + g));
      }
      // ---- dS = P * (scale * dP - scale * D) with P as rounded for the dV product: needs dP^T,
      // which runs after the first half's dV.
      // Its completion also means dK and dQ of the previous step are done with the dS^T buffer.
      ok = mbar_wait(BAR(DP_FULL), n & 1, w, 61);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        continue;
      }
      tc_fence_after();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t col = 64u * g + 32u * r;  // dP^T columns of the quarter
        uint32_t dr[32];
        tmem_ld16(tmem + lane_off + 128 + col, dr);
        tmem_ld16(tmem + lane_off + 128 + col + 16, dr + 16);
        tmem_ld_wait();
        const float4* nd4 = reinterpret_cast<const float4*>(my_dsum + 32 * r);  // -scale * D
        // dS^T row kr, 32 queries = four 16-byte units of the 128-byte swizzled row
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t dd[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int e4 = 2 * u + h;
            const float4 nd = nd4[e4];
            const uint32_t p01 = pp[16 * r + 2 * e4], p23 = pp[16 * r + 2 * e4 + 1];
            // packed f32x2: (scale * dP - scale * D) then times P, the same results as scalar
            float g0, g1, g2, g3;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(p01 << 16), __uint_as_float(p01 & 0xffff0000u)),
                             f2_fma(f2_pack(__uint_as_float(dr[4 * e4 + 0]), __uint_as_float(dr[4 * e4 + 1])), scale2,
                                    f2_pack(nd.x, nd.y))), g0, g1);
            f2_unpack(f2_mul(f2_pack(__uint_as_float(p23 << 16), __uint_as_float(p23 & 0xffff0000u)),
                             f2_fma(f2_pack(__uint_as_float(dr[4 * e4 + 2]), __uint_as_float(dr[4 * e4 + 3])), scale2,
                                    f2_pack(nd.z, nd.w))), g2, g3);
            dd[2 * h] = pack_bf16x2(g0, g1);
            dd[2 * h + 1] = pack_bf16x2(g2, g3);
          }
          *reinterpret_cast<uint4*>(ds_row + (((4 * r + u) ^ swz) << 4)) = make_uint4(dd[0], dd[1], dd[2], dd[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(BAR(DS_READY + 2 * r + g));
      }
    }
    // ------------------------------------------------------------ epilogue: group 0 writes dV, group 1 dK
    if (ok) {
      ok = mbar_wait(BAR(DKV_FINAL), 0, w, 59);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const size_t grow = ((size_t)b_coord * p.n_rows_k + kv_start + kg) * Hkv + h_kv;
        const bool store_ok =
            row_ok && FA_INB(grow * D, grow * D + D - 1, (long long)p.B_tensor * p.n_rows_k * Hkv * D, p.err, 16);
        const uint32_t src = tmem + lane_off + 256u + (g ? (uint32_t)D : 0u);
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(g ? p.dk : p.dv) + grow * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(src + 32 * c, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if (store_ok) {
            if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {  // whole 32-byte sectors per store
              st_global_v8(dst + 32 * c, pk);
              st_global_v8(dst + 32 * c + 16, pk + 8);
            } else {
              uint4* o4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
              for (int i = 0; i < 4; ++i) o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
      }
    }
  } else if (D == 64) {
    // ============================================================ dQ drain, d = 64 (thread = one query row of dQ)
    // warps 0-3 take d columns 0-31, warps 12-15 columns 32-63; float4 atomics into the
    // [B*H][d/4][rows][4] accumulator (a warp's lanes, 32 consecutive rows, cover 512 bytes)
    const int half = warp >= 12 ? 1 : 0;
    const int qw = warp & 3;
    const int qr = qw * 32 + lane;
    const uint32_t src = tmem + ((uint32_t)(qw * 32) << 16) + 384 + 32 * half;
    for (int n = 0; n < n_steps; ++n) {
      float4* acc = reinterpret_cast<float4*>(p.dq_acc) + (size_t)(b_coord * p.H + hq_of(n)) * (D / 4) * p.n_rows;
      const int qg = q_begin + (n % n_q) * 128 + qr;
      bool ok = mbar_wait(BAR(DQ_FULL), n & 1, w, 60);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(src, v);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(BAR(DQ_EMPTY));  // the columns are free for the next dQ
      [[maybe_unused]] const long long acc_base = (long long)(b_coord * p.H + hq_of(n)) * (D / 4) * p.n_rows;
      if (qg < it.q_hi &&  // rows past q_hi see none of this block's keys: their share is zero
          FA_INB(acc_base + (size_t)(8 * half) * p.n_rows + seq_start + qg,
                 acc_base + (size_t)(8 * half + 7) * p.n_rows + seq_start + qg,
                 (long long)p.B_tensor * p.H * (D / 4) * p.n_rows, p.err, 14)) {
        const size_t row = (size_t)seq_start + qg;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          atomicAdd(acc + (size_t)(8 * half + j) * p.n_rows + row,
                    make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
      }
    }
  } else {
    // ============================================================ dQ drain (thread = one d row of dQ^T)
    // warps 0-3 take query columns 0-63, warps 12-15 columns 64-127; each
    // releases its columns right after reading them, before its atomics
    const int half = warp >= 12 ? 1 : 0;
    const int qw = warp & 3;
    const int dr = qw * 32 + lane;
    const uint32_t src = tmem + ((uint32_t)(qw * 32) << 16) + 128 + 64 * half;
    for (int n = 0; n < n_steps; ++n) {
      float* acc = p.dq_acc + row_base_of(hq_of(n)) * D + dr;  // [B*H][rows][d]: a warp's lanes cover 128 bytes
      const int q0 = q_begin + (n % n_q) * 128 + 64 * half;
      int nq = min(64, it.q_hi - q0);  // rows past q_hi see none of this block's keys
      const long long acc_first = (long long)row_base_of(hq_of(n)) * D + dr + (long long)q0 * D;
      if (nq > 0 && !FA_INB(acc_first, acc_first + (long long)(nq - 1) * D, (long long)p.B_tensor * p.H * p.n_rows * D,
                            p.err, 15))
        nq = 0;
      bool ok = mbar_wait(BAR(DQ_FULL), n & 1, w, 60);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(src, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(src + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(BAR(DQ_EMPTY));  // the columns are free for the next dP^T
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j < nq) atomicAdd(acc + (size_t)(q0 + j) * D, __uint_as_float(v[j]));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int MASK>
static auto main_kernel_for() {
  return fa_bwd_main_ov_kernel<D, MASK>;
}

template <int D, int MASK>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  // row tiles: one CTA per (batch, head) and 64 rows
  const long long tiles = (long long)p.B_tensor * p.H * ((p.n_rows + kRowTile - 1) / kRowTile);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  fa_bwd_pre_kernel<D><<<(unsigned)tiles, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(p.o), static_cast<const __nv_bfloat16*>(p.dout), p.lse, p.dsum, p.lse2,
      p.dq_acc, p.H, p.n_rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  auto kern = main_kernel_for<D, MASK>();
  constexpr uint32_t smem = Bwd128Layout<D>::kBytes;
  // set on every launch: the attribute belongs to the current device's context
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // CTAs walk (batch, K/V head) pairs, or K/V heads with an item list
  const int bh = p.num_items > 0 ? p.H / p.kv_group : p.B * (p.H / p.kv_group);
  const int gx = bh < kBwdHeadGroup ? bh : kBwdHeadGroup;
  dim3 grid(gx, p.num_items > 0 ? p.num_items : p.num_kblocks, (bh + gx - 1) / gx);
  kern<<<grid, kBwd128Threads, smem, stream>>>(tq, tk, tv, tdo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  fa_bwd_post_kernel<D><<<(unsigned)tiles, 256, 0, stream>>>(p.dq_acc, static_cast<__nv_bfloat16*>(p.dq), p.H,
                                                             p.n_rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const BwdParams& p, int D, int mask, cudaStream_t stream) {
#define FA_BWD_CASE(DD, MM) \
  if (D == DD && mask == MM) return launch_bwd_t<DD, MM>(tq, tk, tv, tdo, p, stream);
  FA_BWD_CASE(64, kMaskNone)
  FA_BWD_CASE(64, kMaskRight)
  FA_BWD_CASE(64, kMaskWindow)
  FA_BWD_CASE(128, kMaskNone)
  FA_BWD_CASE(128, kMaskRight)
  FA_BWD_CASE(128, kMaskWindow)
#undef FA_BWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

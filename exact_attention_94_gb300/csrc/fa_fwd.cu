// Forward kernel: exact attention with an online softmax on the fifth-generation
// tensor cores (tcgen05) of sm_103a.
//
// Method ("13.14 FlashAttention: IO-aware exact attention", sections "Tile
// decomposition" and "Online softmax"; FlashAttention-2 and its Blackwell
// successor in "efficient-attention/flash-2-3"):
//   for each block of 128 query rows Q_i, sweep the key/value blocks K_j, V_j:
//     S = Q_i K_j^T                      (tensor cores, fp32 in Tensor Memory)
//     m_new = max(m_ref, rowmax(S) * scale * log2 e)
//     if m_new > m_ref + tau: O~ *= 2^(m_ref - m_new), l *= same, m_ref = m_new
//     P = 2^(S * scale * log2 e - m_ref)  (bf16, written back over S in TMEM)
//     l += rowsum(P);  O~ += P V_j         (tensor cores, A operand from TMEM)
//   O = O~ / l,  lse = (m_ref + log2 l) * ln 2.
// The conditional rescale ("And on Blackwell") keeps a stale reference
// maximum until the true maximum has grown by more than 2^tau; l and O~ share
// the reference, so the final division cancels it and the result is exact.
// Masks (causal, sliding window) are bottom-right aligned: query i of a
// sequence with Nq queries and Nk keys sits at key position i + Nk - Nq and
// sees keys [i + Nk - Nq - w_left, i + Nk - Nq + w_right] ("efficient-attention/
// flash-2-3", "Using it, the real way": FlashAttention kernels handle causal masks and sliding windows
// natively; tiles outside every row's window are never visited, the
// block-sparse skipping that FlexAttention's block mask performs).
// rowmax(S) comes with the TMEM load of S: the reducing form of tcgen05.ld
// (sm_103a) returns each thread's largest value beside the values; only the
// rows of a partly masked tile take the maximum again after masking.
// Part of the exponentials may be evaluated on the FMA pipe as
// 2^floor(x) * p3(x - floor(x)) with a cubic fitted in fit_exp2_poly.py: one
// column pair in POLYK (template argument; 0 = none) goes to the cubic.
//
// CTA organisation (one CTA per couple of 256-row query chunks of one head,
// each chunk a pair of 128-row query tiles, computed one after the other):
//   warp 0      TMA producer: Q tiles once, then K_j, V_j into a ring of slots
//   warp 1      allocates TMEM and runs the MMA loop; an elect.sync lane issues each tcgen05.mma
//   warps 4-7   softmax of query tile 0 (thread = row = TMEM lane)
//   warps 8-11  softmax of query tile 1
// The tensor pipe alternates between the two tiles (S0_j, PV1_{j-1}, S1_j,
// PV0_j, ...) so one tile's softmax overlaps the other tile's products.
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [256+d,256+2d).
// d = 128: P overwrites S as bf16 pairs, so a tile's next S waits for its P V.
// d = 64 (bf16): P has columns of its own, P0 [384,448), P1 [448,512), and a
// tile's next S is issued as soon as its softmax has read the current S; the
// order per key tile j is S0_j, S1_j, PV0_{j-1}, PV1_{j-1}.
#include "fa_internal.h"
#include "ptx.cuh"

#include <cmath>

namespace fa {

#ifdef FA_COUNT_RESCALES
// Test builds only (never the product library): rescales taken per (batch,
// head), counted as the tiled model of the oracle counts them: a row's
// reference maximum moves while an earlier one existed.
constexpr int kCountSlots = 4096;
__device__ unsigned long long g_rescale_count[kCountSlots];
#endif

namespace {

template <int D, bool F8>
struct FwdLayout {
  static constexpr uint32_t kElt = F8 ? 1u : 2u;     // bytes per element
  static constexpr uint32_t kTile = 128u * D * kElt; // one 128-row tile (a 128-key V^T tile for e4m3)
  static constexpr uint32_t kChunk = 128u * 128u;    // 128 rows x 128 bytes (one 128-byte swizzle column)
  static constexpr int kStages = (F8 || D == 64) ? 8 : 4;  // K/V ring slots
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = 2 * kTile;
  static constexpr uint32_t kBarOff = kKVOff + kStages * kTile;
  static constexpr uint32_t kBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
};

constexpr int kThreads = 384;
constexpr int kHeadGroup = 8;  // heads whose CTAs are scheduled together

}  // namespace

template <int D, int MASK, int POLYK, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdLayout<D, F8>;
  constexpr bool MASKED = MASK != kMaskNone;
  constexpr bool LEFT = MASK == kMaskWindow;  // rows' keys may start after key 0
  constexpr bool SEPP = D == 64 && !F8;       // P in TMEM columns of its own
  constexpr int NS = L::kStages;
  constexpr int CH = (int)(D * L::kElt / 128);  // 128-byte swizzle columns per row
  constexpr int CHUNK_ELEMS = (int)(128 / L::kElt);
  constexpr uint32_t TILE = L::kTile;
  constexpr uint32_t CHUNK = L::kChunk;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);

  const int warp = warp_id();
  const int lane = lane_id();

  // ---------------------------------------------------------------- work
  // A CTA computes one 256-row query chunk (a pair of 128-row tiles) of one
  // (sequence, head), or, when p.couple is set, two: chunks P-1-u and u of a
  // sequence with P chunks, one after the other, the second one's Q loading
  // while the first one's last products run and the first one's epilogue
  // overlapping the second one's first scores.  Single chunks go heaviest
  // first (chunk P-1-u for CTA u), which packs the tail of a causal grid
  // best; couples halve the CTAs' start and end costs where those weigh more
  // (short or unmasked sequences).  grid: x = head within a group, y = u, z =
  // group of heads (the block scheduler walks x fastest, so the CTAs in flight
  // share a few heads' K/V in L2).  Packed batches with an item list: y
  // enumerates the (sequence, u) items that exist and x, z the heads, so no
  // CTA is launched for the chunks a short sequence does not have.
  int b, h, u;
  if (p.num_items > 0) {
    h = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (h >= p.H) return;
    int units, total;
    const bool found =
        varlen_item(p.cu_seqlens, p.bh_total / p.H, p.couple ? 512 : 256, (int)blockIdx.y, b, u, units, total);
    if (blockIdx.y == gridDim.y - 1 && h == 0 && total > (int)gridDim.y && threadIdx.x == 0 && p.err != nullptr)
      atomicCAS(p.err, 0u, FA_DEVERR_BAD_SEQLEN);  // more items than the grid: the offsets are not as declared
    if (!found) return;
  } else {
    const int bh = (int)(blockIdx.z * gridDim.x + blockIdx.x);
    if (bh >= p.bh_total) return;
    b = bh / p.H;
    h = bh % p.H;
    u = (int)blockIdx.y;
  }
  const int h_kv = h / p.kv_group;  // grouped-query attention: K/V head shared by kv_group query heads
  int seq_start = 0, seq_len = p.seq_len, kv_start = 0, kv_len = p.seq_len_k, b_coord = b;
  if (p.cu_seqlens != nullptr) {
    if (!FA_INB(b, b + 1, p.bh_total / p.H + 1, p.err, 1)) return;  // uniform for the CTA
    seq_start = p.cu_seqlens[b];
    seq_len = p.cu_seqlens[b + 1] - seq_start;
    kv_start = p.cu_seqlens_k[b];
    kv_len = p.cu_seqlens_k[b + 1] - kv_start;
    b_coord = 0;
    if (seq_start < 0 || seq_len < 0 || seq_start > p.n_rows - seq_len || kv_start < 0 || kv_len < 0 ||
        kv_start > p.n_rows_k - kv_len || seq_len > p.max_len || kv_len > p.max_len_k) {
      // offsets outside the tensors, or a sequence longer than the stated maximum: report, touch nothing
      if (threadIdx.x == 0 && p.err != nullptr) atomicCAS(p.err, 0u, FA_DEVERR_BAD_SEQLEN);
      return;
    }
  }
  const int n_chunks = (seq_len + 255) / 256;
  if (u >= (p.couple ? (n_chunks + 1) / 2 : n_chunks)) return;  // uniform for the CTA, before any shared state
  const int n_items = (!p.couple || n_chunks - 1 - u == u) ? 1 : 2;
  auto chunk_of = [&](int it) { return it == 0 ? n_chunks - 1 - u : u; };

  // Key tiles query tile t of chunk `chunk` visits: [lo_t, hi_t).  A tile's rows
  // see keys [key_lo(first row), key_hi(last row)) between them (both bounds
  // grow with the row), so the tiles outside that range are skipped entirely.
  // The producer streams the union of the two tiles' ranges, which is
  // contiguous (tile 1 starts no later than tile 0 ends: window_left +
  // window_right >= 0).
  auto ranges_of = [&](int chunk, int& lo0, int& hi0, int& lo1, int& hi1, int& jmin, int& jmax) {
    int lo_t[2], hi_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r0 = chunk * 256 + 128 * t;
      lo_t[t] = hi_t[t] = 0;
      if (r0 < seq_len) {
        const int r1 = min(r0 + 127, seq_len - 1);
        const int lo = LEFT ? mask_key_lo(r0, seq_len, kv_len, p.win_left) : 0;
        const int hi = MASKED ? mask_key_hi(r1, seq_len, kv_len, p.win_right) : kv_len;
        if (hi > lo) {
          lo_t[t] = lo / 128;
          hi_t[t] = (hi + 127) / 128;
        }
      }
    }
    lo0 = lo_t[0], hi0 = hi_t[0], lo1 = lo_t[1], hi1 = hi_t[1];
    const bool live0 = hi0 > lo0, live1 = hi1 > lo1;
    jmin = live0 ? lo0 : lo1;
    jmax = live1 ? hi1 : hi0;
  };

  // ---------------------------------------------------------------- barriers
  // Per chunk: Q_FULL (Q landed), Q_EMPTY (its last S product done: the Q
  // buffer is free), O_FINAL[t] (tile t's last P V product done; only chunks
  // where tile t sees keys), O_EMPTY[t] (tile t's epilogue has read O).  Per
  // visited key tile: S_FULL[t], P_FULL[t], and the K/V ring's FULL/EMPTY
  // slots, whose counts continue from one chunk to the next.
  // With P in columns of its own (d = 64): S_FREE[t] (the softmax has read
  // S_t: the next S_t may be issued), P_EMPTY[t] (the P V product has read P_t).
  enum { Q_FULL = 0, Q_EMPTY = 1, KV_FULL = 2, KV_EMPTY = 2 + NS, S_FULL = 2 + 2 * NS, P_FULL = S_FULL + 2,
         O_FINAL = P_FULL + 2, O_EMPTY = O_FINAL + 2, S_FREE = O_EMPTY + 2, P_EMPTY = S_FREE + 2,
         DRAIN = P_EMPTY + 2, NBARS = DRAIN + 1 };
  static_assert(8 * NBARS + 8 <= 256, "barrier area");
  const uint32_t bar0 = base + L::kBarOff;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + L::kBarOff + 8 * NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(BAR(Q_FULL), 1);
    mbar_init(BAR(Q_EMPTY), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(BAR(KV_FULL + i), 1);
      mbar_init(BAR(KV_EMPTY + i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(S_FULL + t), 1);
      mbar_init(BAR(P_FULL + t), 128);
      mbar_init(BAR(O_FINAL + t), 1);
      mbar_init(BAR(O_EMPTY + t), 128);
      mbar_init(BAR(S_FREE + t), 128);
      mbar_init(BAR(P_EMPTY + t), 1);
    }
    mbar_init(BAR(DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx w{abort_flag, p.timeout_ns, p.err};

  const uint32_t q_s = base + L::kQOff;
  const uint32_t kv_s = base + L::kKVOff;

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      bool ok = true;
      int ring = 0;  // K/V ring positions used by earlier chunks
      for (int it = 0; it < n_items && ok; ++it) {
        const int q0 = chunk_of(it) * 256;
        int lo0, hi0, lo1, hi1, jmin, jmax;
        ranges_of(chunk_of(it), lo0, hi0, lo1, hi1, jmin, jmax);
        // the previous chunk's S products must be done with the Q buffer
        if (it > 0 && !(ok = mbar_wait(BAR(Q_EMPTY), (it - 1) & 1, w, 9))) break;
        mbar_arrive_expect_tx(BAR(Q_FULL), 2 * TILE);
        for (int t = 0; t < 2; ++t)
          for (int c = 0; c < CH; ++c)
            tma_load_4d(q_s + t * TILE + c * CHUNK, &tm_q, BAR(Q_FULL), c * CHUNK_ELEMS, seq_start + q0 + 128 * t, h,
                        b_coord);
        for (int j = jmin; j < jmax && ok; ++j) {
          for (int which = 0; which < 2; ++which) {
            const int uu = ring + 2 * (j - jmin) + which;
            const int slot = uu % NS;
            if (uu >= NS && !mbar_wait(BAR(KV_EMPTY + slot), ((uu / NS) - 1) & 1, w, 1)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(BAR(KV_FULL + slot), TILE);
            if (F8 && which) {  // V^T codes: d rows of 128 keys
              tma_load_4d(kv_s + slot * TILE, &tm_v, BAR(KV_FULL + slot), 128 * j, 0, h_kv, b_coord);
              continue;
            }
            const CUtensorMap* m = which ? &tm_v : &tm_k;
            for (int c = 0; c < CH; ++c)
              tma_load_4d(kv_s + slot * TILE + c * CHUNK, m, BAR(KV_FULL + slot), c * CHUNK_ELEMS,
                          kv_start + 128 * j, h_kv, b_coord);
          }
        }
        ring += 2 * (jmax - jmin);
      }
      if (!ok) {  // let copies already in flight land before the CTA's shared memory goes away
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    // the whole warp runs the loop; one elected lane issues each product and commit
    {
      constexpr uint32_t IDESC_S = F8 ? idesc_e4m3(128, 128) : idesc_bf16(128, 128, false, false);
      constexpr uint32_t IDESC_O = F8 ? idesc_e4m3(128, D) : idesc_bf16(128, D, false, true);
      const uint32_t tS0 = tmem, tS1 = tmem + 128;
      const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;
      bool ok = true;

      // S_t = Q_t K^T: both operands K-major, 128-byte swizzle; each instruction
      // covers 32 bytes of K (16 bf16 or 32 e4m3 elements)
      auto issue_S = [&](int t, int slot) {
        const uint32_t qa = q_s + t * TILE, ka = kv_s + slot * TILE;
        const uint32_t dst = t ? tS1 : tS0;
        // e4m3: descriptors built once and advanced by an add (measured 1.4% faster there;
        // no difference for bf16)
        [[maybe_unused]] const uint64_t qd = smem_desc_sw128(qa, 16, 1024), kd = smem_desc_sw128(ka, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < (int)(D * L::kElt / 32); ++kk) {
          const uint32_t off = (kk / 4) * CHUNK + (kk % 4) * 32;
          if constexpr (F8)
            mma_ss_f8_w(dst, desc_add(qd, off), desc_add(kd, off), IDESC_S, kk > 0);
          else
            mma_ss_w(dst, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024), IDESC_S, kk > 0);
        }
      };
      // O_t += P_t V with P from TMEM over S_t's columns.  bf16: pairs per column,
      // V MN-major; e4m3: four per column, V^T K-major (d rows of 128 keys).
      auto issue_PV = [&](int t, int slot, bool acc) {
        const uint32_t va = kv_s + slot * TILE;
        const uint32_t dst = t ? tO1 : tO0;
        const uint32_t pa = SEPP ? tmem + 384u + 64u * t : (t ? tS1 : tS0);
        if constexpr (F8) {
          const uint64_t vd = smem_desc_sw128(va, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_f8_w(dst, pa + kk * 8, desc_add(vd, kk * 32), IDESC_O, (acc || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_w(dst, pa + kk * 8, smem_desc_sw128(va + kk * 2048, CHUNK, 1024), IDESC_O,
                   (acc || kk > 0) ? 1u : 0u);
        }
      };

      int ring = 0;                 // K/V ring positions used by earlier chunks
      int sph0 = 0, sph1 = 0;       // S / P phases of each tile used by earlier chunks
      // The first P V product of tile t of chunk `it` overwrites O_t: the previous
      // chunk's epilogue must have read it.
      auto first_pv_ready = [&](int it, int t) -> bool {
        if (it == 0) return true;
        const bool good = __all_sync(0xffffffffu, mbar_wait(BAR(O_EMPTY + t), (it - 1) & 1, w, 10));
        if (good) tc_fence_after();
        return good;
      };
      if constexpr (SEPP) {
        // Per key tile j: S0_j, S1_j (each once its softmax has read the tile's
        // previous S), then PV0_{j-1}, PV1_{j-1} (each once its P has landed).
        int gs[2] = {0, 0};  // S products issued per tile so far (all chunks)
        int gp[2] = {0, 0};  // P V products issued per tile so far
        for (int it = 0; it < n_items && ok; ++it) {
          int lo[2], hi[2], jmin, jmax;
          ranges_of(chunk_of(it), lo[0], hi[0], lo[1], hi[1], jmin, jmax);
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(Q_FULL), it & 1, w, 2)))) break;
          tc_fence_after();
          for (int j = jmin; j <= jmax && ok; ++j) {
            if (j < jmax) {
              const int uk = ring + 2 * (j - jmin), sk = uk % NS;
              if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_FULL + sk), (uk / NS) & 1, w, 3)))) break;
              tc_fence_after();
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (j < lo[t] || j >= hi[t]) continue;
                if (gs[t] > 0) {
                  if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(S_FREE + t), (gs[t] - 1) & 1, w, 11)))) break;
                  tc_fence_after();
                }
                issue_S(t, sk);
                mma_commit_w(BAR(S_FULL + t));
                ++gs[t];
              }
              if (!ok) break;
              if (j == jmax - 1) mma_commit_w(BAR(Q_EMPTY));  // the chunk's last S product
              mma_commit_w(BAR(KV_EMPTY + sk));
            }
            if (j > jmin) {
              const int uv = ring + 2 * (j - 1 - jmin) + 1, sv = uv % NS;
              if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_FULL + sv), (uv / NS) & 1, w, 5)))) break;
              tc_fence_after();
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (j - 1 < lo[t] || j - 1 >= hi[t]) continue;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(P_FULL + t), gp[t] & 1, w, 6)))) break;
                tc_fence_after();
                if (j - 1 == lo[t] && !(ok = first_pv_ready(it, t))) break;
                issue_PV(t, sv, j - 1 > lo[t]);
                mma_commit_w(BAR(P_EMPTY + t));
                if (j - 1 == hi[t] - 1) mma_commit_w(BAR(O_FINAL + t));
                ++gp[t];
              }
              if (!ok) break;
              mma_commit_w(BAR(KV_EMPTY + sv));
            }
          }
          if (ok && jmax <= jmin) mma_commit_w(BAR(Q_EMPTY));  // a chunk with no key tile: nothing read Q
          ring += 2 * (jmax - jmin);
        }
      }
      for (int it = 0; it < n_items && ok && !SEPP; ++it) {
        int jlo0, jhi0, jlo1, jhi1, jmin, jmax;
        ranges_of(chunk_of(it), jlo0, jhi0, jlo1, jhi1, jmin, jmax);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(Q_FULL), it & 1, w, 2)))) break;
        tc_fence_after();
        // Ring position u of key tile j is ring + 2 (j - jmin) (K) and + 1 (V);
        // tile t's S / P barriers complete once per visited key tile.
        for (int j = jmin; j < jmax && ok; ++j) {
          const int uk = ring + 2 * (j - jmin), sk = uk % NS;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_FULL + sk), (uk / NS) & 1, w, 3)))) break;
          tc_fence_after();
          if (j >= jlo0 && j < jhi0) {
            issue_S(0, sk);
            mma_commit_w(BAR(S_FULL + 0));
          }
          if (j > jmin) {
            const int sv = (uk - 1) % NS;
            if (j - 1 >= jlo1 && j - 1 < jhi1) {
              if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(P_FULL + 1), (sph1 + j - 1 - jlo1) & 1, w, 4))))
                break;
              tc_fence_after();
              if (j - 1 == jlo1 && !(ok = first_pv_ready(it, 1))) break;
              issue_PV(1, sv, j - 1 > jlo1);
              if (j - 1 == jhi1 - 1) mma_commit_w(BAR(O_FINAL + 1));
            }
            mma_commit_w(BAR(KV_EMPTY + sv));
          }
          if (j >= jlo1 && j < jhi1) {
            issue_S(1, sk);
            mma_commit_w(BAR(S_FULL + 1));
          }
          // the chunk's last S product: the Q buffer is free once it is done
          if (j == jmax - 1) mma_commit_w(BAR(Q_EMPTY));
          mma_commit_w(BAR(KV_EMPTY + sk));
          const int uv = uk + 1, sv = uv % NS;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(KV_FULL + sv), (uv / NS) & 1, w, 5)))) break;
          tc_fence_after();
          if (j >= jlo0 && j < jhi0) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(BAR(P_FULL + 0), (sph0 + j - jlo0) & 1, w, 6))))
              break;
            tc_fence_after();
            if (j == jlo0 && !(ok = first_pv_ready(it, 0))) break;
            issue_PV(0, sv, j > jlo0);
            if (j == jhi0 - 1) mma_commit_w(BAR(O_FINAL + 0));
          }
        }
        if (ok && jmax > jmin) {
          const int j = jmax;
          const int sv = (ring + 2 * (j - 1 - jmin) + 1) % NS;
          if (j - 1 >= jlo1 && j - 1 < jhi1) {
            if ((ok = __all_sync(0xffffffffu, mbar_wait(BAR(P_FULL + 1), (sph1 + j - 1 - jlo1) & 1, w, 4)))) {
              tc_fence_after();
              if (j - 1 == jlo1) ok = first_pv_ready(it, 1);
              if (ok) {
                issue_PV(1, sv, j - 1 > jlo1);
                mma_commit_w(BAR(O_FINAL + 1));
              }
            }
          }
          if (ok) mma_commit_w(BAR(KV_EMPTY + sv));
        }
        if (ok && jmax <= jmin) mma_commit_w(BAR(Q_EMPTY));  // a chunk with no key tile: nothing read Q
        ring += 2 * (jmax - jmin);
        sph0 += jhi0 - jlo0;
        sph1 += jhi1 - jlo1;
      }
      // Drain: every product and every earlier commit's arrival has landed
      // before TMEM is released and the CTA's shared memory goes away.
      mma_commit_w(BAR(DRAIN));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(BAR(DRAIN), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
      }
    }
  } else if (warp >= 4) {
    // ============================================================ softmax
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (t ? 128u : 0u);
    const uint32_t tO = tmem + lane_off + 256u + (t ? (uint32_t)D : 0u);
    const uint32_t tP = SEPP ? tmem + lane_off + 384u + 64u * (uint32_t)t : tS;  // where P goes
    const float sl2 = p.scale_log2;
    const float tau = p.tau;
#ifdef FA_COUNT_RESCALES
    const int bh_count = b * p.H + h;
#endif
    bool ok = true;
    // e4m3 operands: scores of key tile j are dequantised by sq (this query
    // tile's scale) * sk_j; P of tile j is multiplied by sv_j / sv_ref before
    // its rounding to e4m3 (sv_ref = the head's largest V scale, so P stays in
    // [0, 2^tau]) and O by sv_ref at the end.  The factor goes into the
    // exponent, and l adds P back at its own scale.
    float sv_ref = 1.f;
    const float* k_sc = nullptr;
    const float* v_sc = nullptr;
    [[maybe_unused]] const long long n_kv_scales = (long long)(p.bh_total / p.H) * (p.H / p.kv_group) * p.n_kblk;
    const long long hk = (long long)b * (p.H / p.kv_group) + h_kv;
    if constexpr (F8) {
      k_sc = p.k_scale + hk * p.n_kblk;
      v_sc = p.v_scale + hk * p.n_kblk;
      float mv = 0.f;
      for (int i = lane; i < p.n_kblk; i += 32)
        if (FA_INB(hk * p.n_kblk + i, hk * p.n_kblk + i, n_kv_scales, p.err, 5)) mv = fmaxf(mv, v_sc[i]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
      sv_ref = mv > 0.f ? mv : 1.f;
    }
    int sphase = 0;  // S / P phases of this tile used by earlier chunks
    int nfinal = 0;  // O_FINAL phases of this tile used by earlier chunks
    for (int it = 0; it < n_items && ok; ++it) {
      const int q0 = chunk_of(it) * 256;
      int lo0, hi0, lo1, hi1, jmin_, jmax_;
      ranges_of(chunk_of(it), lo0, hi0, lo1, hi1, jmin_, jmax_);
      const int row = q0 + 128 * t + r;
      float m_ref = -INFINITY;
      float l = 0.f;
      // keys this row sees: [key_lo, key_hi)
      const int key_lo = LEFT ? mask_key_lo(row, seq_len, kv_len, p.win_left) : 0;
      const int key_hi = MASKED ? mask_key_hi(row, seq_len, kv_len, p.win_right) : kv_len;
      const int jlo = t ? lo1 : lo0, jhi = t ? hi1 : hi0;
      float sl2_q = sl2;
      if constexpr (F8) {
        const int qb = (q0 >> 7) + t;  // past the last block only when this tile has no rows
        const size_t qsi = ((size_t)b * p.H + h) * p.n_qblk + qb;
        sl2_q = (qb < p.n_qblk && FA_INB(qsi, qsi, (long long)p.bh_total * p.n_qblk, p.err, 6)) ? sl2 * p.q_scale[qsi]
                                                                                               : 0.f;
      }

      for (int j = jlo; j < jhi; ++j) {
        float sl2j = sl2, lrv = 0.f, inv_rv = 1.f;
        if constexpr (F8) {
          // an all-zero Q or K block (scale 0) has all-zero codes, so its scores are
          // exactly 0 under any positive multiplier; a positive one keeps masked
          // -inf scores at -inf instead of turning them into NaN
          const bool sc_ok = FA_INB(hk * p.n_kblk + j, hk * p.n_kblk + j, n_kv_scales, p.err, 7);
          sl2j = fmaxf(sl2_q * (sc_ok ? k_sc[j] : 0.f), 1e-30f);
          const float rv = fmaxf((sc_ok ? v_sc[j] : 0.f) / sv_ref, 0x1p-30f);  // a zero block's P rounds to 0 either way
          lrv = log2f(rv);
          inv_rv = 1.f / rv;
        }
        ok = mbar_wait(BAR(S_FULL + t), (sphase + j - jlo) & 1, w, 7);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[4][32];
        float mq[4];  // each load's maximum over its 32 columns
  #pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_max(tS + 32 * c, sr[c], mq[c]);
        tmem_ld_wait();
        float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        if constexpr (SEPP) {  // S is in registers: the tile's next S may be issued
          tc_fence_before();
          mbar_arrive(BAR(S_FREE + t));
        }
        float x[128];
  #pragma unroll
        for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(sr[i / 32][i % 32]);

        const int kv0 = 128 * j;
        if ((LEFT && kv0 < key_lo) || kv0 + 128 > key_hi) {
          // a tile the row sees only in part: mask, then take the maximum again
          // (eight short chains of 3-input maxima, then a small tree)
  #pragma unroll
          for (int i = 0; i < 128; ++i)
            if ((LEFT && kv0 + i < key_lo) || kv0 + i >= key_hi) x[i] = -INFINITY;
          float mg[8];
  #pragma unroll
          for (int g = 0; g < 8; ++g) {
            float m = fmaxf(x[16 * g], x[16 * g + 1]);
  #pragma unroll
            for (int i = 2; i < 16; i += 2) m = max3f(m, x[16 * g + i], x[16 * g + i + 1]);
            mg[g] = m;
          }
          mx = max3f(max3f(mg[0], mg[1], mg[2]), max3f(mg[3], mg[4], mg[5]), fmaxf(mg[6], mg[7]));
        }
        const float m_new = mx * sl2j;
        float alpha = 1.f;
        const bool resc = m_new > m_ref + tau;
  #ifdef FA_COUNT_RESCALES
        if (resc && m_ref > -INFINITY && row < seq_len && bh_count < kCountSlots)
          atomicAdd(&g_rescale_count[bh_count], 1ull);
  #endif
        if (resc) {
          alpha = ex2_sfu(m_ref - m_new);
          m_ref = m_new;
        }
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
        if constexpr (SEPP) {
          // the previous P V product of this tile must have read P (and be done
          // adding into O, which a rescale below multiplies)
          const int g = sphase + j - jlo;
          if (g > 0) {
            ok = mbar_wait(BAR(P_EMPTY + t), (g - 1) & 1, w, 12);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
        }

        // p = 2^(x * scale * log2 e - m_ref): packed FMA, exponentials, packed partial sums
        const uint64_t sl2x2 = f2_pack(sl2j, sl2j);
        const uint64_t nmb2 = f2_pack(lrv - mb, lrv - mb);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[2][32];
        float ph0 = 0.f, ph1 = 0.f;  // e4m3: the previous pair, packed with the next into one word
  #pragma unroll
        for (int i = 0; i < 64; ++i) {
          float y0, y1;
          f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), sl2x2, nmb2), y0, y1);
          float p0, p1;
          if (POLYK > 0 && (i % (POLYK > 0 ? POLYK : 1)) == POLYK - 1) {
            ex2_poly2(y0, y1, p0, p1);
          } else {
            p0 = ex2_sfu(y0);
            p1 = ex2_sfu(y1);
          }
          acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
          if constexpr (F8) {
            if (i & 1)
              pk[0][i / 2] = pack_e4m3x4(ph0, ph1, p0, p1);  // keys 4c..4c+3 in column c
            else
              ph0 = p0, ph1 = p1;
          } else {
            pk[i / 32][i % 32] = pack_bf16x2(p0, p1);
            if (i == 31) tmem_st32(tP, pk[0]);  // first half of P out early: frees registers
          }
        }
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2_unpack(acc[0], s0, s1);
        f2_unpack(acc[1], s2, s3);
        f2_unpack(acc[2], s4, s5);
        f2_unpack(acc[3], s6, s7);
        l = l * alpha + (((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7))) * inv_rv;

        if (j > jlo && __any_sync(0xffffffffu, resc)) {
          // rows whose reference moved: O~ *= alpha (alpha = 1 for the others)
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + 32 * c, ov);
            tmem_ld_wait();
  #pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tO + 32 * c, ov);
          }
        }
        if constexpr (F8)
          tmem_st32(tS, pk[0]);  // the whole tile's P: 32 columns of four e4m3 each
        else
          tmem_st32(tP + 32, pk[1]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(P_FULL + t));
      }
      sphase += jhi - jlo;
      if (!ok) break;
      // ---------------------------------------------------------- epilogue of the chunk
      const long long o_off = (((long long)b_coord * p.n_rows + seq_start + row) * p.H + h) * D;
      const long long l_off = ((long long)b_coord * p.H + h) * p.n_rows + seq_start + row;
      [[maybe_unused]] const long long b_tensor = p.cu_seqlens != nullptr ? 1 : p.bh_total / p.H;
      const bool row_ok = row < seq_len &&
                          FA_INB(o_off, o_off + D - 1, b_tensor * p.n_rows * p.H * D, p.err, 2) &&
                          FA_INB(l_off, l_off, b_tensor * p.H * p.n_rows, p.err, 3);
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + o_off;
      float* lse_out = p.lse + l_off;
      if (jhi <= jlo) {
        // no key tile visible to any row of this tile: O = 0, lse = -inf
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
          *lse_out = -INFINITY;
        }
      } else {
        ok = mbar_wait(BAR(O_FINAL + t), nfinal & 1, w, 8);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ++nfinal;
        tc_fence_after();
        const float inv_l = l > 0.f ? sv_ref / l : 0.f;  // sv_ref = 1 unless e4m3
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tO + 32 * c, ov);
          tmem_ld_wait();
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
          if (row_ok) {
            if ((reinterpret_cast<uintptr_t>(orow) & 31) == 0) {  // whole 32-byte sectors per store
              st_global_v8(orow + 32 * c, pkd);
              st_global_v8(orow + 32 * c + 16, pkd + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
            }
          }
        }
        if (row_ok) *lse_out = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
      // O has been read: the next chunk's first P V product may overwrite it
      tc_fence_before();
      mbar_arrive(BAR(O_EMPTY + t));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int MASK, int POLYK, bool F8>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, int grid_x, cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, MASK, POLYK, F8>;
  constexpr uint32_t smem = FwdLayout<D, F8>::kBytes;
  // The shared-memory limit is a function attribute of the current device's
  // context; it is set on every launch (no cached per-device state to go stale
  // or to race on between host threads).
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // grid_x: (batch, head) units, or heads with an item list
  const int gx = grid_x < kHeadGroup ? grid_x : kHeadGroup;
  // y: 256-row query chunks (or couples of them), or the packed batch's items
  dim3 grid(gx, p.num_items > 0 ? p.num_items : (p.couple ? (p.num_pairs + 1) / 2 : p.num_pairs),
            (grid_x + gx - 1) / gx);
  kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                       int D, int mask, int poly, int grid_x, cudaStream_t stream) {
#define FA_FWD_CASE(DD, MM, PP) \
  if (D == DD && mask == MM && poly == PP) return launch_fwd_t<DD, MM, PP, false>(tq, tk, tv, p, grid_x, stream);
  // the cubic's share is selectable (1/4, 1/8, 1/16 of the column pairs) for
  // the unmasked and causal kernels; the windowed ones take 1/8, 1/16 or none
#define FA_FWD_CASES(DD)            \
  FA_FWD_CASE(DD, kMaskNone, 0)     \
  FA_FWD_CASE(DD, kMaskNone, 4)     \
  FA_FWD_CASE(DD, kMaskNone, 8)     \
  FA_FWD_CASE(DD, kMaskNone, 16)    \
  FA_FWD_CASE(DD, kMaskRight, 0)    \
  FA_FWD_CASE(DD, kMaskRight, 4)    \
  FA_FWD_CASE(DD, kMaskRight, 8)    \
  FA_FWD_CASE(DD, kMaskRight, 16)   \
  FA_FWD_CASE(DD, kMaskWindow, 0)   \
  FA_FWD_CASE(DD, kMaskWindow, 8)   \
  FA_FWD_CASE(DD, kMaskWindow, 16)
  FA_FWD_CASES(64)
  FA_FWD_CASES(128)
#undef FA_FWD_CASES
#undef FA_FWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const FwdParams& p,
                           int mask, int poly, int grid_x, cudaStream_t stream) {
#define FA_FP8_CASE(MM, PP) \
  if (mask == MM && poly == PP) return launch_fwd_t<128, MM, PP, true>(tq, tk, tvt, p, grid_x, stream);
  FA_FP8_CASE(kMaskNone, 0)
  FA_FP8_CASE(kMaskNone, 8)
  FA_FP8_CASE(kMaskNone, 16)
  FA_FP8_CASE(kMaskRight, 0)
  FA_FP8_CASE(kMaskRight, 8)
  FA_FP8_CASE(kMaskRight, 16)
  FA_FP8_CASE(kMaskWindow, 0)
  FA_FP8_CASE(kMaskWindow, 8)
#undef FA_FP8_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

#ifdef FA_COUNT_RESCALES
// Test builds only: copies out (and clears) the per-(batch, head) rescale counts.
extern "C" int fa_test_rescale_counts(unsigned long long* host, int n) {
  if (n < 0 || n > fa::kCountSlots) return 1;
  if (cudaMemcpyFromSymbol(host, fa::g_rescale_count, sizeof(unsigned long long) * n) != cudaSuccess) return 2;
  static const unsigned long long zeros[fa::kCountSlots] = {};
  return cudaMemcpyToSymbol(fa::g_rescale_count, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 3;
}
#endif

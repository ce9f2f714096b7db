// Single-token decode with a split KV cache (Flash-Decoding).
//
// Method ("efficient-attention/flash-2-3", "Decoding needs a different
// split"): with one query per sequence there is nothing to parallelise over
// but the keys, so the cache is cut into chunks; each chunk yields its own
// normalised output O_c and log-sum-exp lse_c, and a small second kernel
// merges them as the mass-weighted average
//     lse = log sum_c e^(lse_c),   O = sum_c e^(lse_c - lse) O_c.
//
// The step is bound by HBM: every key and value of the cache is read once
// (2*B*L*H*d*2 bytes) for about one FLOP per byte, so the kernel is built
// around keeping enough bytes in flight, not around the tensor cores (one
// query row would waste them).
//
// Split kernel: one CTA per (chunk, batch entry, group of up to 32 heads).
// The cache layout [B, L, H, d] puts one key's heads next to each other, so
// a stage of T keys for the group is T contiguous runs of G*d elements,
// fetched by one producer lane with plain bulk copies into a ring of shared
// memory.  Eight compute warps own 4 heads each; lane i holds d/32 elements
// of the query, of the output accumulator and of every key/value row it
// reads.  Dot products of 4 keys are reduced together with a halving
// butterfly (6 shuffles for 4 keys instead of 20), then an online-softmax
// update in registers (base 2, scale folded into the query).
#include "fa_internal.h"
#include "ptx.cuh"

#include <cmath>

namespace fa {

namespace {

constexpr int kDecT = 4;            // keys per stage
constexpr int kDecWarps = 8;        // compute warps
constexpr int kDecThreads = 32 * (kDecWarps + 1);  // + one producer warp
constexpr int kDecMaxG = 32;        // heads per CTA
constexpr int kDecHPW = kDecMaxG / kDecWarps;      // heads per compute warp

__device__ __forceinline__ void bf16x4_to_f32(uint2 u, float* f) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16* src, float* f) {
  if constexpr (E == 4) {
    bf16x4_to_f32(*reinterpret_cast<const uint2*>(src), f);
  } else {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src));
    f[0] = a.x;
    f[1] = a.y;
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kDecThreads, 1) fa_decode_split_kernel(const DecodeParams p) {
  constexpr int E = D / 32;  // elements per lane
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 127u) & ~127u;
  uint8_t* sbase = smem_raw + (base - raw);

  const int warp = warp_id();
  const int lane = lane_id();
  const int c = blockIdx.x;   // chunk
  const int b = blockIdx.y;   // batch entry
  const int hg = blockIdx.z;  // group of K/V heads
  const int G = p.G;                 // K/V heads of this CTA
  const int Gq = G * p.kv_group;     // query heads of this CTA (those K/V heads' groups)
  const int NS = p.stages;
  const uint32_t row_bytes = (uint32_t)G * D * 2;         // one key, all heads of the group
  const uint32_t stage_bytes = 2u * kDecT * row_bytes;    // K rows then V rows
  int L_b = p.L;  // keys of this sequence
  if (p.seq_lens != nullptr) {
    L_b = p.seq_lens[b];
    if (L_b < 0 || L_b > p.L) {  // never read past what the caller described
      if (threadIdx.x == 0) atomicCAS(p.err, 0u, FA_DEVERR_BAD_SEQLEN);
      L_b = L_b < 0 ? 0 : p.L;
    }
  }
  // a sliding window keeps the last win_left + 1 keys: the splits cover [kbeg, L_b)
  const int kbeg = p.win_left >= 0 ? max(0, L_b - 1 - p.win_left) : 0;
  const int l0 = kbeg + c * p.chunk;
  const int l1 = min(L_b, l0 + p.chunk);
  const int n_keys = max(0, l1 - l0);
  const int n_st = (n_keys + kDecT - 1) / kDecT;

  const uint32_t bar0 = base + (uint32_t)NS * stage_bytes;
  auto FULL = [&](int s) -> uint32_t { return bar0 + 8u * (uint32_t)s; };
  auto EMPTY = [&](int s) -> uint32_t { return bar0 + 8u * (uint32_t)(NS + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + NS * stage_bytes + 16 * NS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), kDecWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx w{abort_flag, p.timeout_ns, p.err};
  const size_t kv_head0 = (size_t)hg * G * D;

  if (warp == kDecWarps) {
    // ============================================================ producer
    if (lane == 0) {
      bool ok = true;
      // paged: the key's logical block and slot, advanced key by key; the block
      // table is read once per page, when the walk enters it
      int pblk = 0, pslot = 0, page = 0;
      auto lookup = [&]() {
        const size_t ti = (size_t)b * p.max_blocks + pblk;
        page = FA_INB(ti, ti, (long long)p.B * p.max_blocks, p.err, 20) ? p.block_table[ti] : 0;
        if (page < 0 || page >= p.num_pages) {  // report, and read a valid page instead
          atomicCAS(p.err, 0u, FA_DEVERR_BAD_PAGE);
          page = 0;
        }
      };
      if (p.block_table != nullptr && n_keys > 0) {
        pblk = l0 / p.page_size;
        pslot = l0 - pblk * p.page_size;
        lookup();
      }
      for (int s = 0; s < n_st && ok; ++s) {
        const int slot = s % NS;
        if (s >= NS && !(ok = mbar_wait(EMPTY(slot), ((s / NS) - 1) & 1, w, 41))) break;
        const int nv = min(kDecT, n_keys - s * kDecT);
        mbar_arrive_expect_tx(FULL(slot), 2u * nv * row_bytes);
        const uint32_t dk = base + slot * stage_bytes;
        for (int m = 0; m < nv; ++m) {
          const int l = l0 + s * kDecT + m;
          size_t row;
          if (p.block_table != nullptr) {  // paged: logical block -> physical page
            row = ((size_t)page * p.page_size + pslot) * p.Hkv * D + kv_head0;
            if (++pslot == p.page_size) {
              pslot = 0;
              ++pblk;
              if (l + 1 < l1) lookup();  // the next key lies on the next page
            }
          } else {
            row = ((size_t)b * p.L + l) * p.Hkv * D + kv_head0;
          }
          // (bounds-checked builds: a row outside the cache is reported and the group's row 0 read instead,
          // so that the stage's byte count still completes)
          if (!FA_INB(row, row + (size_t)G * D - 1,
                      p.block_table != nullptr ? (long long)p.num_pages * p.page_size * p.Hkv * D
                                               : (long long)p.B * p.L * p.Hkv * D,
                      p.err, 21))
            row = kv_head0;
          bulk_load(dk + m * row_bytes, static_cast<const __nv_bfloat16*>(p.k) + row, row_bytes, FULL(slot));
          bulk_load(dk + (kDecT + m) * row_bytes, static_cast<const __nv_bfloat16*>(p.v) + row, row_bytes,
                    FULL(slot));
        }
      }
      if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else {
    // ============================================================ compute warps
    float qv[kDecHPW][E], o[kDecHPW][E], m_run[kDecHPW], l_lane[kDecHPW];
    int kv_off[kDecHPW];  // element offset of this lane's slice of its K/V head within a staged key row
#pragma unroll
    for (int j = 0; j < kDecHPW; ++j) {
      const int hj = warp + kDecWarps * j;
      kv_off[j] = (hj / p.kv_group) * D + lane * E;
      m_run[j] = -INFINITY;
      l_lane[j] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[j][e] = 0.f;
      const size_t q_off = ((size_t)b * p.H + hg * Gq + hj) * D + lane * E;
      if (hj < Gq && FA_INB(q_off, q_off + E - 1, (long long)p.B * p.H * D, p.err, 22)) {
        const __nv_bfloat16* qs = static_cast<const __nv_bfloat16*>(p.q) + q_off;
        load_row<E>(qs, qv[j]);
#pragma unroll
        for (int e = 0; e < E; ++e) qv[j][e] *= p.scale_log2;  // scores come out in log2 units
      }
    }
    // lane -> key slot after the butterfly: bit 4 picks the pair, bit 3 the key in it
    const int my_key = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
    bool ok = true;
    for (int s = 0; s < n_st; ++s) {
      const int slot = s % NS;
      ok = mbar_wait(FULL(slot), (s / NS) & 1, w, 42);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const int nv = min(kDecT, n_keys - s * kDecT);
      const __nv_bfloat16* ks = reinterpret_cast<const __nv_bfloat16*>(sbase + slot * stage_bytes);
      const __nv_bfloat16* vs = ks + kDecT * G * D;
#pragma unroll
      for (int j = 0; j < kDecHPW; ++j) {
        const int hj = warp + kDecWarps * j;  // query head of the CTA
        if (hj >= Gq) break;
        // partial dot products of this lane's elements for the 4 keys
        float part[kDecT];
#pragma unroll
        for (int m = 0; m < kDecT; ++m) {
          float kf[E];
          load_row<E>(ks + m * G * D + kv_off[j], kf);
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) acc = fmaf(qv[j][e], kf[e], acc);
          part[m] = acc;
        }
        // halving butterfly: after it every lane holds the full score of key my_key
        const bool up = lane & 16;
        const float a0 = (up ? part[2] : part[0]) + __shfl_xor_sync(0xffffffffu, up ? part[0] : part[2], 16);
        const float a1 = (up ? part[3] : part[1]) + __shfl_xor_sync(0xffffffffu, up ? part[1] : part[3], 16);
        const bool b8 = lane & 8;
        float sc = (b8 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, b8 ? a0 : a1, 8);
        sc += __shfl_xor_sync(0xffffffffu, sc, 4);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        if (my_key >= nv) sc = -INFINITY;
        float mb = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 8));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
        const float m_new = fmaxf(m_run[j], mb);
        const float alpha = (m_new == -INFINITY) ? 1.f : ex2_sfu(m_run[j] - m_new);
        const float pm = (m_new == -INFINITY) ? 0.f : ex2_sfu(sc - m_new);
        l_lane[j] = fmaf(l_lane[j], alpha, pm);
        m_run[j] = m_new;
#pragma unroll
        for (int e = 0; e < E; ++e) o[j][e] *= alpha;
#pragma unroll
        for (int m = 0; m < kDecT; ++m) {
          if (m < nv) {
            const float pk = __shfl_sync(0xffffffffu, pm, (m >> 1) * 16 + (m & 1) * 8);
            float vf[E];
            load_row<E>(vs + m * G * D + kv_off[j], vf);
#pragma unroll
            for (int e = 0; e < E; ++e) o[j][e] = fmaf(pk, vf[e], o[j][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(slot));
    }
    // ------------------------------------------------------------ partial results
    if (ok) {
#pragma unroll
      for (int j = 0; j < kDecHPW; ++j) {
        const int hj = warp + kDecWarps * j;
        if (hj >= Gq) break;
        float l = l_lane[j] + __shfl_xor_sync(0xffffffffu, l_lane[j], 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const size_t pidx = ((size_t)b * p.H + hg * Gq + hj) * p.num_splits + c;
        if (!FA_INB(pidx, pidx, (long long)p.B * p.H * p.num_splits, p.err, 23)) continue;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* dst = p.part_o + pidx * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = o[j][e] * inv;
        if (lane == 0) p.part_lse[pidx] = l > 0.f ? m_run[j] + __log2f(l) : -INFINITY;
      }
    }
  }
}

// Log-sum-exp merge of the chunks' partial results; one warp per (batch, head).
// Partials are in base 2: part_lse = log2 of the chunk's softmax mass (scale included).
template <int D>
__global__ void __launch_bounds__(256) fa_decode_combine_kernel(const float* __restrict__ part_o,
                                                               const float* __restrict__ part_lse,
                                                               __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                               int BH, int S) {
  constexpr int E = D / 32;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= BH) return;
  const float* pl = part_lse + (size_t)gw * S;
  float m = -INFINITY;
  for (int c = lane; c < S; c += 32) m = fmaxf(m, pl[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int c = 0; c < S; ++c) {
      const float wc = ex2_sfu(pl[c] - m);  // an empty chunk has lse = -inf: weight 0
      wsum += wc;
      const float* src = part_o + ((size_t)gw * S + c) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(wc, src[e], acc[e]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = o + (size_t)gw * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const uint32_t pk = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + e) = pk;
  }
  if (lane == 0) lse[gw] = wsum > 0.f ? (m + __log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

int decode_stages(int G, int D) {
  const int stage = 2 * kDecT * G * D * 2;
  int ns = (192 * 1024) / stage;
  return ns < 2 ? 2 : (ns > 8 ? 8 : ns);
}

size_t decode_smem_bytes(int G, int D) {
  const int ns = decode_stages(G, D);
  return (size_t)ns * 2 * kDecT * G * D * 2 + 16 * ns + 16 + 128;
}

template <int D>
static cudaError_t launch_decode_t(const DecodeParams& p, void* o, float* lse, cudaStream_t stream) {
  auto kern = fa_decode_split_kernel<D>;
  const size_t smem = decode_smem_bytes(p.G, D);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_splits, p.B, p.Hkv / p.G);
  kern<<<grid, kDecThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int bh = p.B * p.H;
  fa_decode_combine_kernel<D><<<(bh + 7) / 8, 256, 0, stream>>>(p.part_o, p.part_lse,
                                                                static_cast<__nv_bfloat16*>(o), lse, bh,
                                                                p.num_splits);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int D, void* o, float* lse, cudaStream_t stream) {
  if (D == 64) return launch_decode_t<64>(p, o, lse, stream);
  if (D == 128) return launch_decode_t<128>(p, o, lse, stream);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- paged cache: append
//
// One CTA per appended token: copy page copy_src -> page first when the
// token's sequence shared a partly filled last page, then write the token's
// K and V rows into its slot.  Sequences that still share a page all sit at
// the same length, so a copy that overlaps another holder's in-place write
// only reads the slot this CTA overwrites next.
__global__ void __launch_bounds__(256) fa_paged_append_kernel(const uint4* __restrict__ k_new,
                                                              const uint4* __restrict__ v_new, uint4* k_pages,
                                                              uint4* v_pages, const int* __restrict__ page,
                                                              const int* __restrict__ slot,
                                                              const int* __restrict__ copy_src, int row_vec,
                                                              int page_size, int num_pages, unsigned* err) {
  const int i = blockIdx.x;
  const int pg = page[i], sl = slot[i], src = copy_src[i];
  if (pg < 0 || pg >= num_pages || sl < 0 || sl >= page_size || src >= num_pages) {
    if (threadIdx.x == 0) atomicCAS(err, 0u, FA_DEVERR_BAD_PAGE);
    return;
  }
  const size_t page_vec = (size_t)page_size * row_vec;  // 16-byte vectors per page
  if (src >= 0) {
    const uint4* ks = k_pages + (size_t)src * page_vec;
    const uint4* vs = v_pages + (size_t)src * page_vec;
    uint4* kd = k_pages + (size_t)pg * page_vec;
    uint4* vd = v_pages + (size_t)pg * page_vec;
    for (size_t t = threadIdx.x; t < page_vec; t += blockDim.x) {
      kd[t] = ks[t];
      vd[t] = vs[t];
    }
    __syncthreads();
  }
  uint4* kd = k_pages + (size_t)pg * page_vec + (size_t)sl * row_vec;
  uint4* vd = v_pages + (size_t)pg * page_vec + (size_t)sl * row_vec;
  for (int t = threadIdx.x; t < row_vec; t += blockDim.x) {
    kd[t] = k_new[(size_t)i * row_vec + t];
    vd[t] = v_new[(size_t)i * row_vec + t];
  }
}

cudaError_t launch_paged_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages, const int* page,
                                const int* slot, const int* copy_src, int n, int Hkv, int d, int page_size,
                                int num_pages, unsigned* err, cudaStream_t stream) {
  const int row_vec = Hkv * d / 8;  // bf16 x 8 per vector
  fa_paged_append_kernel<<<n, 256, 0, stream>>>(static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                                                static_cast<uint4*>(k_pages), static_cast<uint4*>(v_pages), page, slot,
                                                copy_src, row_vec, page_size, num_pages, err);
  return cudaGetLastError();
}

}  // namespace fa

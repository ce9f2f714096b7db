// Block quantisation of Q, K, V to e4m3 for the FP8 forward pass, with
// optional incoherent processing ("efficient-attention/flash-2-3", section
// "FP8, and the outlier problem": one scale per block of Q, K and V, the
// blocks the kernel loads anyway; Q and K multiplied by the same Hadamard
// matrix times a random +-1 diagonal before quantising).
//
// One CTA per 128-row block of one (batch, head); warp w owns rows
// 8w .. 8w+7, a row is spread over d/16 lanes of 16 consecutive columns.
//   rotate:   x <- (x H) * signs, H the Sylvester-Hadamard matrix (entries
//             +-1), by the fast transform: stage widths 1, 2, 4, ..., d/2, each
//             butterfly (a, b) -> (a + b, a - b) in fp32.  Widths below 16
//             stay inside a lane, the others pair lanes with shuffles.  The
//             signs are applied in the final multiply by the inverse scale.
//   scale:    amax / 448 over the block (fp32, correctly rounded); 0 for an
//             all-zero block, whose codes are 0.
//   codes:    e4m3(x * (1 / scale)), the reciprocal and the product each
//             correctly rounded, the conversion rounding to nearest even and
//             saturating.
//   layout:   codes [B][N][H][d] like the input, or (V) transposed per head,
//             [B][H][d][n_pad], n_pad = blocks * 128, rows past N zero, so
//             that the P V product reads V^T K-major.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kQuantThreads = 512;  // 16 warps; each takes 8 rows of the 128-row block
constexpr int kRowsPerWarp = kQuantThreads == 512 ? 8 : 16;
constexpr int kElems = 16;          // consecutive elements per lane

// Butterflies of widths 1 .. 8 inside the lane's 16 elements, then widths
// 16 * hl with the lane that differs in bit hl (hl < lanes per row).  The
// elements are held as eight fp32 pairs: width 1 pairs the two halves of a
// pair (scalar), widths 2 .. 8 and the cross-lane stages use the packed
// f32x2 add, subtract and FMA, which round exactly like the scalar ones.
template <int LPR>
__device__ __forceinline__ void fwht_row16(uint64_t (&vp)[kElems / 2], int lane) {
#pragma unroll
  for (int i = 0; i < kElems / 2; ++i) {
    float a, b;
    f2_unpack(vp[i], a, b);
    vp[i] = f2_pack(a + b, a - b);
  }
#pragma unroll
  for (int h = 1; h < kElems / 2; h <<= 1) {
#pragma unroll
    for (int i = 0; i < kElems / 2; ++i) {
      if (!(i & h)) {
        const uint64_t a = vp[i], b = vp[i + h];
        vp[i] = f2_add(a, b);
        vp[i + h] = f2_sub(a, b);
      }
    }
  }
  // the lower lane of a pair keeps a + b, the upper one a - b: one FMA with a
  // +-1 multiplier, rounded once exactly like the add or subtract it replaces
#pragma unroll
  for (int hl = 1; hl < LPR; hl <<= 1) {
    const float sg = (lane & hl) ? -1.f : 1.f;
    const uint64_t sg2 = f2_pack(sg, sg);
#pragma unroll
    for (int i = 0; i < kElems / 2; ++i) {
      float lo, hi;
      f2_unpack(vp[i], lo, hi);
      lo = __shfl_xor_sync(0xffffffffu, lo, hl);
      hi = __shfl_xor_sync(0xffffffffu, hi, hl);
      vp[i] = f2_fma(vp[i], sg2, f2_pack(lo, hi));
    }
  }
}

}  // namespace

template <int D, bool ROT, bool TR>
__global__ void __launch_bounds__(kQuantThreads) fa_fp8_quant_kernel(const __nv_bfloat16* __restrict__ x,
                                                                     const int8_t* __restrict__ signs,
                                                                     uint8_t* __restrict__ codes,
                                                                     float* __restrict__ scales, int N, int H,
                                                                     int nblk) {
  constexpr int LPR = D / kElems;   // lanes per row
  constexpr int RPI = 32 / LPR;     // rows per warp and iteration
  constexpr int IT = kRowsPerWarp / RPI;  // iterations over the warp's rows
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = lane % LPR;       // which 16 columns of the row
  const int sub = lane / LPR;       // which row of the iteration
  __shared__ float s_amax[kQuantThreads / 32];
  __shared__ __align__(16) uint8_t s_rows[TR ? 128 * D : 16];  // codes, row-major, for the transposed store

  uint32_t neg = 0;  // bit e: column seg*16 + e takes the sign -1
  if (ROT) {
#pragma unroll
    for (int e = 0; e < kElems; ++e) neg |= (signs[seg * kElems + e] < 0 ? 1u : 0u) << e;
  }

  uint64_t v[IT][kElems / 2];  // pairs of fp32 elements
  float amax = 0.f;
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int n = blk * 128 + warp * kRowsPerWarp + it * RPI + sub;
    if (n < N) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (((size_t)b * N + n) * H + h) * D + seg * kElems);
      const uint4 w0 = src[0], w1 = src[1];
      const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[it][i] = f2_pack(__uint_as_float(wv[i] << 16), __uint_as_float(wv[i] & 0xffff0000u));
    } else {
#pragma unroll
      for (int i = 0; i < kElems / 2; ++i) v[it][i] = 0ull;
    }
    if (ROT) fwht_row16<LPR>(v[it], lane);  // the signs come with the scale below
#pragma unroll
    for (int i = 0; i < kElems / 2; ++i) {
      float a, b;
      f2_unpack(v[it][i], a, b);
      amax = max3f(amax, fabsf(a), fabsf(b));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_amax[warp] = amax;
  __syncthreads();
  amax = s_amax[0];
#pragma unroll
  for (int i = 1; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, s_amax[i]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  const float inv = amax > 0.f ? __frcp_rn(scale) : 0.f;  // codes = e4m3(x * (1 / scale))
  if (threadIdx.x == 0) scales[((size_t)b * H + h) * nblk + blk] = scale;
  // x * sign * (1 / scale) as x * (sign * (1 / scale)): the sign is exact and
  // round-to-nearest is symmetric, so each code (and each zero's sign) is the same
  uint64_t sinv[kElems / 2];
#pragma unroll
  for (int i = 0; i < kElems / 2; ++i)
    sinv[i] = f2_pack(((neg >> (2 * i)) & 1u) ? -inv : inv, ((neg >> (2 * i + 1)) & 1u) ? -inv : inv);

#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int rr = warp * kRowsPerWarp + it * RPI + sub;  // row within the block
    const int n = blk * 128 + rr;
    uint32_t wd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float y0, y1, y2, y3;
      f2_unpack(f2_mul(v[it][2 * q], sinv[2 * q]), y0, y1);
      f2_unpack(f2_mul(v[it][2 * q + 1], sinv[2 * q + 1]), y2, y3);
      wd[q] = pack_e4m3x4(y0, y1, y2, y3);
    }
    uint4 word = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    if (!(amax > 0.f)) word = make_uint4(0u, 0u, 0u, 0u);  // all-zero block: +0 codes (not -0 from flipped zeros)
    if constexpr (TR) {
      if (n >= N) word = make_uint4(0u, 0u, 0u, 0u);  // padding rows: +0 (a rotated zero row would give -0)
      *reinterpret_cast<uint4*>(s_rows + rr * D + seg * kElems) = word;
    } else if (n < N) {
      *reinterpret_cast<uint4*>(codes + (((size_t)b * N + n) * H + h) * D + seg * kElems) = word;
    }
  }
  if constexpr (TR) {
    // thread -> column c, half of the rows: gather 64 bytes of column c and
    // write them as one contiguous run of row c of V^T
    __syncthreads();
    const size_t n_pad = (size_t)nblk * 128;
    for (int i = threadIdx.x; i < D * 2; i += kQuantThreads) {
      const int c = i % D, half = i / D;
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int r0 = half * 64 + 4 * k;
        w[k] = (uint32_t)s_rows[r0 * D + c] | ((uint32_t)s_rows[(r0 + 1) * D + c] << 8) |
               ((uint32_t)s_rows[(r0 + 2) * D + c] << 16) | ((uint32_t)s_rows[(r0 + 3) * D + c] << 24);
      }
      uint4* dst = reinterpret_cast<uint4*>(codes + (((size_t)b * H + h) * D + c) * n_pad + (size_t)blk * 128 +
                                            half * 64);
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
  }
}

cudaError_t launch_fp8_quantize(const void* x, const int8_t* signs, uint8_t* codes, float* scales, int B, int N,
                                int H, int d, bool rotate, bool transpose, cudaStream_t stream) {
  const int nblk = (N + 127) / 128;
  dim3 grid(nblk, H, B);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
#define FA_QUANT_CASE(DD, RR, TT)                                                                       \
  if (d == DD && rotate == RR && transpose == TT) {                                                     \
    fa_fp8_quant_kernel<DD, RR, TT><<<grid, kQuantThreads, 0, stream>>>(xb, signs, codes, scales, N, H, nblk); \
    return cudaGetLastError();                                                                          \
  }
  FA_QUANT_CASE(128, true, false)
  FA_QUANT_CASE(128, false, false)
  FA_QUANT_CASE(128, false, true)
  FA_QUANT_CASE(128, true, true)
  FA_QUANT_CASE(64, true, false)
  FA_QUANT_CASE(64, false, false)
  FA_QUANT_CASE(64, false, true)
  FA_QUANT_CASE(64, true, true)
#undef FA_QUANT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa

// Block quantisation of Q, K, V to e4m3 for the FP8 forward pass, with
// optional incoherent processing ("efficient-attention/flash-2-3", section
// "FP8, and the outlier problem": one scale per block of Q, K and V, the
// blocks the kernel loads anyway; Q and K multiplied by the same Hadamard
// matrix times a random +-1 diagonal before quantising).
//
// One CTA per 128-row block of one (batch, head); warp w owns rows
// 16w .. 16w+15, lane l the d/32 consecutive columns l*d/32 ... of each row.
//   rotate:   x <- (x H) * signs, H the Sylvester-Hadamard matrix (entries
//             +-1), by the fast transform: stage widths 1, 2, 4, ..., d/2, each
//             butterfly (a, b) -> (a + b, a - b) in fp32.  Widths below d/32
//             stay inside a lane, the others pair lanes with shuffles.
//   scale:    amax / 448 over the block (fp32, correctly rounded); 0 for an
//             all-zero block, whose codes are 0.
//   codes:    e4m3(x / scale), the division correctly rounded, the conversion
//             rounding to nearest even and saturating.
//   layout:   codes [B][N][H][d] like the input, or (V) transposed per head,
//             [B][H][d][n_pad], n_pad = blocks * 128, rows past N zero, so
//             that the P V product reads V^T K-major.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kQuantThreads = 256;
constexpr int kRowsPerWarp = 16;

template <int E>
__device__ __forceinline__ void fwht_row(float (&v)[E], int lane) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (!(i & h)) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int hl = 1; hl < 32; hl <<= 1) {  // width E * hl: the partner lane differs in bit hl
    const bool upper = (lane & hl) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], hl);
      v[i] = upper ? (o - v[i]) : (v[i] + o);
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
  constexpr int E = D / 32;
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float s_amax[kQuantThreads / 32];
  __shared__ __align__(16) uint8_t s_t[TR ? D * 128 : 16];

  float sg[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = ROT ? (float)signs[lane * E + e] : 1.f;

  float v[kRowsPerWarp][E];
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int n = blk * 128 + warp * kRowsPerWarp + r;
    if (n < N) {
      const __nv_bfloat16* src = x + (((size_t)b * N + n) * H + h) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + e));
        v[r][e] = f.x;
        v[r][e + 1] = f.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[r][e] = 0.f;
    }
    if (ROT) {
      fwht_row<E>(v[r], lane);
#pragma unroll
      for (int e = 0; e < E; ++e) v[r][e] *= sg[e];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[r][e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_amax[warp] = amax;
  __syncthreads();
  amax = s_amax[0];
#pragma unroll
  for (int i = 1; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, s_amax[i]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  if (threadIdx.x == 0) scales[((size_t)b * H + h) * nblk + blk] = scale;

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int rr = warp * kRowsPerWarp + r;  // row within the block
    const int n = blk * 128 + rr;
    float y[E];
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = scale > 0.f ? __fdiv_rn(v[r][e], scale) : 0.f;
    uint32_t word;
    if constexpr (E == 4)
      word = pack_e4m3x4(y[0], y[1], y[2], y[3]);
    else
      word = pack_e4m3x4(y[0], y[1], 0.f, 0.f);
    if constexpr (TR) {
      if (n >= N) word = 0u;  // padding rows: +0 (a rotated zero row would give -0 codes)
#pragma unroll
      for (int e = 0; e < E; ++e) s_t[(lane * E + e) * 128 + rr] = (uint8_t)(word >> (8 * e));
    } else if (n < N) {
      uint8_t* dst = codes + (((size_t)b * N + n) * H + h) * D + lane * E;
      if constexpr (E == 4)
        *reinterpret_cast<uint32_t*>(dst) = word;
      else
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)word;
    }
  }
  if constexpr (TR) {
    __syncthreads();
    const size_t n_pad = (size_t)nblk * 128;
    for (int i = threadIdx.x; i < D * 8; i += kQuantThreads) {  // D rows of 128 bytes, 16 bytes each
      const int c = i >> 3, part = i & 7;
      const uint4 val = *reinterpret_cast<const uint4*>(s_t + c * 128 + part * 16);
      *reinterpret_cast<uint4*>(codes + (((size_t)b * H + h) * D + c) * n_pad + (size_t)blk * 128 + part * 16) = val;
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

// C ABI of the library: argument validation, tensor-map construction,
// workspace sizing and kernel launches.  See include/fa.h for the contract of
// every entry point.
#include "../../include/fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

namespace fa {

__device__ unsigned int g_fa_error = 0;
constexpr unsigned kSelftestSite = 0xFFu;

// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// ever arrives on, through the same helper every kernel uses.
__global__ void fa_wait_selftest_kernel(unsigned* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx w{&abort_flag, timeout_ns, err};
  mbar_wait(smem_u32(&bar), 0, w, kSelftestSite);
}

// Evaluates one of the library's exp2 implementations elementwise (self-test);
// each thread takes two neighbouring elements (the packed cubic works on pairs).
__global__ void fa_exp2_selftest_kernel(const float* __restrict__ x, float* __restrict__ y, int n, int which) {
  const long long i = 2ll * (blockIdx.x * (long long)blockDim.x + threadIdx.x);
  if (i >= n) return;
  const bool two = i + 1 < n;
  const float v0 = x[i], v1 = two ? x[i + 1] : 0.f;
  float y0, y1;
  if (which == 0) {
    y0 = ex2_poly(v0);
    y1 = ex2_poly(v1);
  } else if (which == 1) {
    y0 = ex2_sfu(v0);
    y1 = ex2_sfu(v1);
  } else if (which == 2) {
    y0 = exp2f(v0);
    y1 = exp2f(v1);
  } else {
    ex2_poly2(v0, v1, y0, y1);
  }
  y[i] = y0;
  if (two) y[i + 1] = y1;
}

namespace {

struct Options {
  float tau = 8.0f;
  int poly = 16;  // one column pair in `poly` on the cubic (0 = none): measured fastest at d = 64 and 128
  unsigned long long timeout_ns = 2000000000ull;
} g_opt;

std::once_flag g_init_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

thread_local unsigned* g_err_ptr = nullptr;  // the current device's error word, set by ensure_init()

void init_once() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Every entry point calls this before it builds kernel parameters: it resolves
// the driver entry point once per process, and looks up the error word's
// device address on every call, with the caller's device current (the symbol
// has an address of its own on each device, and a new one after the device's
// context is torn down and created again; the lookup allocates nothing).
bool ensure_init() {
  std::call_once(g_init_once, init_once);
  if (g_encode == nullptr) return false;
  void* ep = nullptr;
  if (cudaGetSymbolAddress(&ep, g_fa_error) != cudaSuccess || ep == nullptr) return false;
  g_err_ptr = static_cast<unsigned*>(ep);
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

bool make_tmap_bhnd(CUtensorMap* m, const void* ptr, int D, int n_rows, int H, int B, int box_rows) {
  const cuuint64_t e = 2;  // bytes per bf16
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)n_rows, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)H * D * e, (cuuint64_t)D * e, (cuuint64_t)n_rows * H * D * e};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u8(CUtensorMap* m, const void* ptr, const uint64_t dims_in[4], const uint64_t strides_in[3],
                  int box_y) {
  cuuint64_t dims[4] = {dims_in[0], dims_in[1], dims_in[2], dims_in[3]};
  cuuint64_t strides[3] = {strides_in[0], strides_in[1], strides_in[2]};
  cuuint32_t box[4] = {128, (cuuint32_t)box_y, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_SCRATCH_LIMIT: return "FA_ERR_SCRATCH_LIMIT";
    case FA_ERR_OUT_OF_PAGES: return "FA_ERR_OUT_OF_PAGES";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_set_option(fa_option opt, double value) {
  switch (opt) {
    case FA_OPT_RESCALE_TAU:
      if (!(value >= 0.0 && value <= 64.0)) return FA_ERR_INVALID_ARG;
      g_opt.tau = (float)value;
      return FA_OK;
    case FA_OPT_POLY_EXP:  // 0 = off, 1 = the default share (1/8), or the share's denominator 4, 8, 16
      if (value == 0.0 || value == 4.0 || value == 8.0 || value == 16.0) {
        g_opt.poly = (int)value;
        return FA_OK;
      }
      if (value == 1.0) {
        g_opt.poly = 8;
        return FA_OK;
      }
      return FA_ERR_INVALID_ARG;
    case FA_OPT_WAIT_TIMEOUT_MS:
      if (!(value >= 1.0 && value <= 600000.0)) return FA_ERR_INVALID_ARG;
      g_opt.timeout_ns = (unsigned long long)(value * 1e6);
      return FA_OK;
  }
  return FA_ERR_INVALID_ARG;
}

fa_status fa_selftest_wait_timeout(double timeout_ms, fa_stream_t stream) {
  if (!(timeout_ms >= 1.0 && timeout_ms <= 10000.0)) return FA_ERR_INVALID_ARG;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  fa_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(g_err_ptr, (unsigned long long)(timeout_ms * 1e6));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_selftest_exp2(const float* x, float* y, int n, int which, fa_stream_t stream) {
  if (n < 0 || which < 0 || which > 3 || (n > 0 && (!x || !y))) return FA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 3u) != 0) return FA_ERR_MISALIGNED;
  if (n == 0) return FA_OK;
  const long long pairs = ((long long)n + 1) / 2;
  fa_exp2_selftest_kernel<<<(unsigned)((pairs + 255) / 256), 256, 0, (cudaStream_t)stream>>>(x, y, n, which);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_device_error(unsigned int* code) {
  if (!ensure_init()) return FA_ERR_LAUNCH;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_error, sizeof(v)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (code) *code = v;
  if (v != 0) {
    const unsigned zero = 0;
    cudaMemcpyToSymbol(g_fa_error, &zero, sizeof(zero));
    return v >= FA_DEVERR_BAD_PAGE ? FA_ERR_INVALID_ARG : FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

// Window bounds: -1 leaves a side unbounded; a bound that reaches past every
// key of the longest sequence is the same as none, so it is dropped.
static bool window_ok(int& wl, int& wr, int max_len_q, int max_len_k) {
  if (wl < -1 || wr < -1) return false;
  if (wl >= max_len_k) wl = -1;
  if (wr >= max_len_q) wr = -1;
  return true;
}

// Grid rows of a packed batch's item list: an upper bound of the (sequence,
// unit) items, sum_b ceil(len_b / unit) <= min(num_seqs * ceil(max_len / unit),
// ceil(total / unit) + num_seqs).  0 (no list: the grid covers every sequence's
// max_len) when the bound or the sequence count is too large for it.
static int packed_items(int num_seqs, int units_max, int total_rows, int unit) {
  const long long by_max = (long long)num_seqs * units_max;
  const long long by_total = ((long long)total_rows + unit - 1) / unit + num_seqs;
  const long long items = by_max < by_total ? by_max : by_total;
  if (num_seqs > 2048 || items > 65535 || items < 1) return 0;
  return (int)items;
}

// The bf16 sliding-window kernels exist with the cubic off or on one column
// pair in 8 or 16 (1/4 maps to 1/8).  The e4m3 kernels have 1/8 and none, and
// without a window also 1/16 (the fastest share measured for them); with a
// window 1/16 maps to none.
static int window_poly(int poly) { return poly == 16 ? 16 : (poly == 4 || poly == 8) ? 8 : 0; }
static int fp8_poly(int poly, int mask) {
  if (poly == 16) return mask == kMaskWindow ? 0 : 16;
  return (poly == 4 || poly == 8) ? 8 : 0;
}

static fa_status fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu,
                            const int* cu_k, int nbatch, int n_rows, int n_rows_k, int seq_len, int seq_len_k,
                            int max_len, int max_len_k, int H, int Hkv, int d, int wl, int wr, float scale,
                            fa_stream_t stream) {
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale) || !window_ok(wl, wr, max_len, max_len_k)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  if ((long long)nbatch * H > 65535LL * 8) return FA_ERR_INVALID_ARG;  // grid.z limit with 8-head groups
  const int num_pairs = (max_len + 255) / 256;
  if (num_pairs > 65535) return FA_ERR_INVALID_ARG;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  CUtensorMap tq, tk, tv;
  const int tb = cu ? 1 : nbatch;
  if (!make_tmap_bhnd(&tq, q, d, n_rows, H, tb) || !make_tmap_bhnd(&tk, k, d, n_rows_k, Hkv, tb) ||
      !make_tmap_bhnd(&tv, v, d, n_rows_k, Hkv, tb))
    return FA_ERR_INVALID_ARG;
  FwdParams p{};
  p.kv_group = H / Hkv;
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu;
  p.cu_seqlens_k = cu_k;
  p.H = H;
  p.bh_total = nbatch * H;
  p.n_rows = n_rows;
  p.n_rows_k = n_rows_k;
  p.seq_len = seq_len;
  p.seq_len_k = seq_len_k;
  p.win_left = wl;
  p.win_right = wr;
  p.num_pairs = num_pairs;
  // Couples of chunks per CTA for packed batches and unmasked calls, where the
  // CTAs' start and end costs weigh most; single chunks, heaviest first, for
  // masked dense calls, whose grid tail packs better that way.
  const int mk = mask_kind(wl, wr);
  p.couple = (cu != nullptr || mk == kMaskNone) ? 1 : 0;
  p.num_items = cu ? (p.couple ? packed_items(nbatch, (num_pairs + 1) / 2, n_rows, 512)
                               : packed_items(nbatch, num_pairs, n_rows, 256))
                   : 0;
  p.max_len = max_len;
  p.max_len_k = max_len_k;
  p.scale_log2 = scale * kLog2e;
  p.tau = g_opt.tau;
  p.err = g_err_ptr;
  p.timeout_ns = g_opt.timeout_ns;
  const int poly = mk == kMaskWindow ? window_poly(g_opt.poly) : g_opt.poly;
  cudaError_t e = launch_fwd(tq, tk, tv, p, d, mk, poly, p.num_items > 0 ? H : nbatch * H, (cudaStream_t)stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// causal flag of the square entry points -> window (-1, 0), else no mask
static int causal_right(int causal) { return causal ? 0 : -1; }

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 int causal, float scale, fa_stream_t stream) {
  if (B < 1 || H < 1 || N < 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (N == 0) return FA_OK;
  return fwd_common(q, k, v, o, lse, nullptr, nullptr, B, N, N, N, N, N, N, H, H, d, -1, causal_right(causal),
                    scale, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                     int d, int causal, float scale, fa_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (N == 0) return FA_OK;
  return fwd_common(q, k, v, o, lse, nullptr, nullptr, B, N, N, N, N, N, N, Hq, Hkv, d, -1, causal_right(causal),
                    scale, stream);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                        int num_seqs, int max_seqlen, int total_tokens, int H, int d, int causal, float scale,
                        fa_stream_t stream) {
  if (num_seqs < 1 || H < 1 || max_seqlen < 0 || total_tokens < 0 || !cu_seqlens) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return FA_ERR_MISALIGNED;
  if (total_tokens == 0 || max_seqlen == 0) return FA_OK;
  return fwd_common(q, k, v, o, lse, cu_seqlens, cu_seqlens, num_seqs, total_tokens, total_tokens, 0, 0, max_seqlen,
                    max_seqlen, H, H, d, -1, causal_right(causal), scale, stream);
}

fa_status fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, int window_left, int window_right, float scale, fa_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (Nq == 0) return FA_OK;
  if (Nk == 0) {  // no keys: the kernel writes O = 0 and lse = -inf; K and V are never read
    return fwd_common(q, q, q, o, lse, nullptr, nullptr, B, Nq, 1, Nq, 0, Nq, 1, Hq, Hq, d, -1, -1, scale,
                      stream);
  }
  return fwd_common(q, k, v, o, lse, nullptr, nullptr, B, Nq, Nk, Nq, Nk, Nq, Nk, Hq, Hkv, d, window_left,
                    window_right, scale, stream);
}

fa_status fa_fwd_masked_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs, int max_seqlen_q,
                               int max_seqlen_k, int total_q, int total_k, int Hq, int Hkv, int d, int window_left,
                               int window_right, float scale, fa_stream_t stream) {
  if (num_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  if (max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0) return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k)) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  if (total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (total_k == 0) {  // every sequence has an empty cache: O = 0 and lse = -inf
    return fwd_common(q, q, q, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, 1, 0, 0, max_seqlen_q, 1, Hq,
                      Hq, d, -1, -1, scale, stream);
  }
  if (max_seqlen_k == 0) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, 0, 0, max_seqlen_q,
                    max_seqlen_k, Hq, Hkv, d, window_left, window_right, scale, stream);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 0 || d < 1) return 0;
  const size_t acc = (size_t)B * N * H * d * sizeof(float);  // fp32 dQ accumulator
  const size_t rows = (size_t)B * H * N * sizeof(float);     // D and lse * log2 e
  return align256(acc) + 2 * align256(rows);
}

size_t fa_bwd_varlen_workspace_bytes(int total_tokens, int H, int d) {
  return fa_bwd_workspace_bytes(1, H, total_tokens, d);
}

static fa_status bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, void* workspace, const int* cu,
                            const int* cu_k, int nbatch, int n_rows, int n_rows_k, int seq_len, int seq_len_k,
                            int max_len, int max_len_k, int H, int Hkv, int d, int wl, int wr, float scale,
                            fa_stream_t stream) {
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale) || !window_ok(wl, wr, max_len, max_len_k)) return FA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA_ERR_MISALIGNED;
  if ((long long)nbatch * H > 65535LL * 8) return FA_ERR_INVALID_ARG;
  const int num_kblocks = (max_len_k + 127) / 128;
  if (num_kblocks > 65535) return FA_ERR_INVALID_ARG;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  const int tb = cu ? 1 : nbatch;
  CUtensorMap tq, tk, tv, tdo;
  const int q_box = 128;
  if (!make_tmap_bhnd(&tq, q, d, n_rows, H, tb, q_box) || !make_tmap_bhnd(&tk, k, d, n_rows_k, Hkv, tb) ||
      !make_tmap_bhnd(&tv, v, d, n_rows_k, Hkv, tb) || !make_tmap_bhnd(&tdo, dout, d, n_rows, H, tb, q_box))
    return FA_ERR_INVALID_ARG;
  const size_t acc_bytes = align256((size_t)tb * n_rows * H * d * sizeof(float));
  const size_t row_bytes = align256((size_t)tb * H * n_rows * sizeof(float));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BwdParams p{};
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq_acc = reinterpret_cast<float*>(ws);
  p.dsum = reinterpret_cast<float*>(ws + acc_bytes);
  p.lse2 = reinterpret_cast<float*>(ws + acc_bytes + row_bytes);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.cu_seqlens = cu;
  p.cu_seqlens_k = cu_k;
  p.B = nbatch;
  p.B_tensor = tb;
  p.H = H;
  p.kv_group = H / Hkv;
  p.n_rows = n_rows;
  p.n_rows_k = n_rows_k;
  p.seq_len = seq_len;
  p.seq_len_k = seq_len_k;
  p.win_left = wl;
  p.win_right = wr;
  p.num_kblocks = num_kblocks;
  p.num_items = cu ? packed_items(nbatch, num_kblocks, n_rows_k, 128) : 0;
  p.max_len = max_len;
  p.max_len_k = max_len_k;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.err = g_err_ptr;
  p.timeout_ns = g_opt.timeout_ns;
  cudaError_t e = launch_bwd(tq, tk, tv, tdo, p, d, mask_kind(wl, wr), (cudaStream_t)stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, void* workspace, int B, int H, int N, int d, int causal, float scale,
                 fa_stream_t stream) {
  if (B < 1 || H < 1 || N < 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (N == 0) return FA_OK;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr, nullptr, B, N, N, N, N, N, N, H, H, d,
                    -1, causal_right(causal), scale, stream);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, void* workspace, int B, int Hq, int Hkv, int N, int d, int causal,
                     float scale, fa_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 0 || Hq % Hkv != 0 || (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  if (N == 0) return FA_OK;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr, nullptr, B, N, N, N, N, N, N, Hq, Hkv, d,
                    -1, causal_right(causal), scale, stream);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, const int* cu_seqlens,
                        int num_seqs, int max_seqlen, int total_tokens, int H, int d, int causal, float scale,
                        fa_stream_t stream) {
  if (num_seqs < 1 || H < 1 || max_seqlen < 0 || total_tokens < 0 || !cu_seqlens) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return FA_ERR_MISALIGNED;
  if (total_tokens == 0 || max_seqlen == 0) return FA_OK;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, cu_seqlens, cu_seqlens, num_seqs, total_tokens,
                    total_tokens, 0, 0, max_seqlen, max_seqlen, H, H, d, -1, causal_right(causal), scale, stream);
}

fa_status fa_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, int window_left, int window_right, float scale, fa_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nk < 1 || Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr, nullptr, B, Nq, Nk, Nq, Nk, Nq, Nk, Hq,
                    Hkv, d, window_left, window_right, scale, stream);
}

fa_status fa_bwd_masked_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, void* workspace,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs, int max_seqlen_q,
                               int max_seqlen_k, int total_q, int total_k, int Hq, int Hkv, int d, int window_left,
                               int window_right, float scale, fa_stream_t stream) {
  if (num_seqs < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
  if (max_seqlen_q < 1 || max_seqlen_k < 1 || total_q < 1 || total_k < 1) return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k)) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q,
                    total_k, 0, 0, max_seqlen_q, max_seqlen_k, Hq, Hkv, d, window_left, window_right, scale, stream);
}

// ---------------------------------------------------------------- backward without allocation
//
// Scratch of fa_bwd_noalloc: the fp32 dQ accumulator and the two per-row
// arrays fa_bwd otherwise takes from a caller-allocated workspace.  It is
// part of the library's device image, so every GPU that loads the library
// holds these bytes until the process exits.  All calls share it.
static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                         float scale, fa_stream_t stream) {
  if (B < 1 || H < 1 || N < 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (N == 0) return FA_OK;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (fa_bwd_workspace_bytes(B, H, N, d) > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  // The array's device address, looked up with the caller's device current on
  // every call (in host code the symbol itself is only a stand-in; the lookup
  // allocates nothing, and a context created anew after a device reset gets a
  // new address).
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, g_bwd_scratch) != cudaSuccess || scratch == nullptr) return FA_ERR_LAUNCH;
  // The pre-kernel of the backward zeroes the accumulator part of the scratch
  // and overwrites the per-row arrays, so the previous call's contents never leak.
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, scratch, nullptr, nullptr, B, N, N, N, N, N, N, H, H, d, -1,
                    causal_right(causal), scale, stream);
}

// ---------------------------------------------------------------- FP8 forward

fa_status fa_fp8_quantize(const void* x, const signed char* signs, void* codes, float* scales, int B, int N, int H, int d,
                          int rotate, int transpose, fa_stream_t stream) {
  if (B < 1 || H < 1 || N < 0 || (rotate != 0 && rotate != 1) || (transpose != 0 && transpose != 1))
    return FA_ERR_INVALID_ARG;
  if (!x || !codes || !scales || (rotate && !signs)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;
  if (N == 0) return FA_OK;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  cudaError_t e = launch_fp8_quantize(x, signs, static_cast<uint8_t*>(codes), scales, B, N, H, d, rotate != 0,
                                      transpose != 0, (cudaStream_t)stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_fwd_fp8(const void* q_codes, const void* k_codes, const void* vt_codes, const float* q_scale,
                     const float* k_scale, const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                     int Nk, int d, int window_left, int window_right, int rotated, float scale, fa_stream_t stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 0 || Nk < 1 || (rotated != 0 && rotated != 1))
    return FA_ERR_INVALID_ARG;
  if (!q_codes || !k_codes || !vt_codes || !q_scale || !k_scale || !v_scale || !o || !lse) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  int wl = window_left, wr = window_right;
  if (!scale_ok(scale) || !window_ok(wl, wr, Nq, Nk)) return FA_ERR_INVALID_ARG;
  const void* ptrs[] = {q_codes, k_codes, vt_codes, o, lse};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA_ERR_MISALIGNED;
  if (((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
        reinterpret_cast<uintptr_t>(v_scale)) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  if ((long long)B * Hq > 65535LL * 8) return FA_ERR_INVALID_ARG;
  const int num_pairs = (Nq + 255) / 256;
  if (num_pairs > 65535) return FA_ERR_INVALID_ARG;
  if (Nq == 0) return FA_OK;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  const int n_kblk = (Nk + 127) / 128;
  const uint64_t n_pad = (uint64_t)n_kblk * 128;
  CUtensorMap tq, tk, tvt;
  const uint64_t dq[4] = {(uint64_t)d, (uint64_t)Nq, (uint64_t)Hq, (uint64_t)B};
  const uint64_t sq[3] = {(uint64_t)Hq * d, (uint64_t)d, (uint64_t)Nq * Hq * d};
  const uint64_t dk[4] = {(uint64_t)d, (uint64_t)Nk, (uint64_t)Hkv, (uint64_t)B};
  const uint64_t sk[3] = {(uint64_t)Hkv * d, (uint64_t)d, (uint64_t)Nk * Hkv * d};
  const uint64_t dv[4] = {n_pad, (uint64_t)d, (uint64_t)Hkv, (uint64_t)B};
  const uint64_t sv[3] = {n_pad, n_pad * d, n_pad * d * Hkv};
  if (!make_tmap_u8(&tq, q_codes, dq, sq, 128) || !make_tmap_u8(&tk, k_codes, dk, sk, 128) ||
      !make_tmap_u8(&tvt, vt_codes, dv, sv, d))
    return FA_ERR_INVALID_ARG;
  FwdParams p{};
  p.kv_group = Hq / Hkv;
  p.o = o;
  p.lse = lse;
  p.H = Hq;
  p.bh_total = B * Hq;
  p.n_rows = Nq;
  p.n_rows_k = Nk;
  p.seq_len = Nq;
  p.seq_len_k = Nk;
  p.win_left = wl;
  p.win_right = wr;
  p.num_pairs = num_pairs;
  p.max_len = Nq;
  p.max_len_k = Nk;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.n_qblk = (Nq + 127) / 128;
  p.n_kblk = n_kblk;
  p.scale_log2 = scale * kLog2e / (rotated ? (float)d : 1.f);
  p.tau = g_opt.tau;
  p.err = g_err_ptr;
  p.timeout_ns = g_opt.timeout_ns;
  cudaError_t e = launch_fwd_fp8(tq, tk, tvt, p, mask_kind(wl, wr), fp8_poly(g_opt.poly, mask_kind(wl, wr)), B * Hq,
                                 (cudaStream_t)stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_paged_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages, const int* page,
                          const int* slot, const int* copy_src, int n, int Hkv, int d, int page_size, int num_pages,
                          fa_stream_t stream) {
  if (n < 0 || Hkv < 1 || page_size < 1 || num_pages < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (n == 0) return FA_OK;
  if (!k_new || !v_new || !k_pages || !v_pages || !page || !slot || !copy_src) return FA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages)) return FA_ERR_MISALIGNED;
  if (((reinterpret_cast<uintptr_t>(page) | reinterpret_cast<uintptr_t>(slot) |
        reinterpret_cast<uintptr_t>(copy_src)) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  cudaError_t e = launch_paged_append(k_new, v_new, k_pages, v_pages, page, slot, copy_src, n, Hkv, d, page_size,
                                      num_pages, g_err_ptr, (cudaStream_t)stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

size_t fa_decode_workspace_bytes(int B, int H, int d, int num_splits) {
  if (B < 1 || H < 1 || d < 1 || num_splits < 1) return 0;
  const size_t po = (size_t)B * H * num_splits * d * sizeof(float);
  const size_t pl = (size_t)B * H * num_splits * sizeof(float);
  return ((po + 255) & ~(size_t)255) + ((pl + 255) & ~(size_t)255);
}

// K/V heads handled by one decode CTA: the largest divisor G of Hkv whose
// query heads (G * group) fit the CTA's 32 query-head slots.
static int decode_group(int Hkv, int group) {
  for (int g = Hkv < 32 ? Hkv : 32; g > 1; --g)
    if (Hkv % g == 0 && g * group <= 32) return g;
  return 1;
}

static int auto_splits(int B, int Hkv, int group, int L) {
  if (B < 1 || Hkv < 1 || L <= 0) return 1;
  int dev = 0, n_sm = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const long long ctas_per_split = (long long)B * (Hkv / decode_group(Hkv, group));
  // about eight full waves of one CTA per SM, and at least 256 keys per split
  long long s = (8LL * n_sm + ctas_per_split - 1) / ctas_per_split;
  const long long max_s = (L + 255) / 256;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return (int)s;
}

int fa_decode_num_splits(int B, int H, int L, int d) {
  (void)d;
  return auto_splits(B, H, 1, L);
}

// Common decode path: contiguous cache (block_table == nullptr) or paged cache.
static fa_status decode_common(const void* q, const void* k, const void* v, const int* block_table,
                               const int* seq_lens, int page_size, int num_pages, int max_blocks, void* o, float* lse,
                               int B, int H, int Hkv, int L, int d, int num_splits, void* workspace, float scale,
                               fa_stream_t stream, int win_left = -1) {
  if (!q || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Hkv < 1 || H % Hkv != 0 || L < 0 || num_splits < 0 || win_left < -1) return FA_ERR_INVALID_ARG;
  if (win_left >= L) win_left = -1;  // a window past every key is no window
  const int span = win_left >= 0 ? win_left + 1 : L;  // keys a query sees at most
  const int group = H / Hkv;
  if (group > 32) return FA_ERR_UNSUPPORTED;  // a CTA serves at most 32 query heads
  if (L > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;  // an empty contiguous cache may be null
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, lse, workspace};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return FA_ERR_MISALIGNED;
  const int S = num_splits > 0 ? num_splits : auto_splits(B, Hkv, group, span);
  if (L > 0 && S > span) return FA_ERR_INVALID_ARG;
  const int G = decode_group(Hkv, group);
  if (B > 65535 || Hkv / G > 65535) return FA_ERR_INVALID_ARG;
  if (!ensure_init()) return FA_ERR_LAUNCH;
  const size_t part_bytes = align256((size_t)B * H * S * d * sizeof(float));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.part_o = reinterpret_cast<float*>(ws);
  p.part_lse = reinterpret_cast<float*>(ws + part_bytes);
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.kv_group = group;
  p.L = L;
  p.G = G;
  p.chunk = span > 0 ? (span + S - 1) / S : 0;
  p.win_left = win_left;
  p.num_splits = S;
  p.stages = decode_stages(G, d);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.page_size = page_size;
  p.max_blocks = max_blocks;
  p.num_pages = num_pages;
  p.scale_log2 = scale * kLog2e;
  p.err = g_err_ptr;
  p.timeout_ns = g_opt.timeout_ns;
  cudaError_t e = launch_decode(p, d, o, lse, (cudaStream_t)stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                          const int* seq_lens, void* o, float* lse, int B, int H, int d, int page_size, int num_pages,
                          int max_blocks, int max_seq_len, int num_splits, void* workspace, float scale,
                          fa_stream_t stream) {
  if (!k_pages || !v_pages || !block_table || !seq_lens) return FA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_blocks < 1 || max_seq_len < 0) return FA_ERR_INVALID_ARG;
  if (page_size < 4 || page_size % 4 != 0 || (long long)max_blocks * page_size < max_seq_len)
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return FA_ERR_MISALIGNED;
  return decode_common(q, k_pages, v_pages, block_table, seq_lens, page_size, num_pages, max_blocks, o, lse, B, H, H,
                       max_seq_len, d, num_splits, workspace, scale, stream);
}

fa_status fa_decode_window(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                           int Hkv, int L, int d, int window_left, int num_splits, void* workspace, float scale,
                           fa_stream_t stream) {
  return decode_common(q, k_cache, v_cache, nullptr, nullptr, 0, 0, 0, o, lse, B, Hq, Hkv, L, d, num_splits,
                       workspace, scale, stream, window_left);
}

fa_status fa_decode_paged_window(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                                 const int* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d,
                                 int page_size, int num_pages, int max_blocks, int max_seq_len, int window_left,
                                 int num_splits, void* workspace, float scale, fa_stream_t stream) {
  if (!k_pages || !v_pages || !block_table || !seq_lens) return FA_ERR_INVALID_ARG;
  if (num_pages < 1 || max_blocks < 1 || max_seq_len < 0) return FA_ERR_INVALID_ARG;
  if (page_size < 4 || page_size % 4 != 0 || (long long)max_blocks * page_size < max_seq_len)
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return FA_ERR_MISALIGNED;
  return decode_common(q, k_pages, v_pages, block_table, seq_lens, page_size, num_pages, max_blocks, o, lse, B, Hq,
                       Hkv, max_seq_len, d, num_splits, workspace, scale, stream, window_left);
}

fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B,
                            int H, int L, int d, int num_splits, void* workspace, float scale, fa_stream_t stream) {
  return decode_common(q, k_cache, v_cache, nullptr, nullptr, 0, 0, 0, o, lse, B, H, H, L, d, num_splits, workspace,
                       scale, stream);
}

fa_status fa_decode_gqa(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                        int Hkv, int L, int d, int num_splits, void* workspace, float scale, fa_stream_t stream) {
  return decode_common(q, k_cache, v_cache, nullptr, nullptr, 0, 0, 0, o, lse, B, Hq, Hkv, L, d, num_splits,
                       workspace, scale, stream);
}

}  // extern "C"

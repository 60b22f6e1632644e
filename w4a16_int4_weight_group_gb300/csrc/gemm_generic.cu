// Generic W4A16 product for any shape the layer allows (N % 8 == 0, any K, natural alignment only).
//
// Each CTA owns 32 packed words (256 output columns) and 8 rows of A. Its 256 threads are 32 word
// columns x 8 K-slices: thread (c, s) walks k = s, s+8, s+16, ..., dequantises the word b_q[k, c]
// into eight values RNE_dtype((q - zp) * scale) - exactly the values w4a16_dequant materialises - and
// accumulates A[m, k] * w in fp32 for its 8 rows. The 8 K-slices are summed in shared memory in a
// fixed order, bias is added in fp32, and the result is rounded once to the activation dtype
// (PR #40977 report, key source snippets, test reference: bias added before the cast).
// This path exists for shapes and pointers the fast paths cannot take; it favours simplicity.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kCols = 32;    // packed words per CTA
constexpr int kSlices = 8;   // K slices per CTA
constexpr int kRows = 8;     // rows of A per CTA

template <class DT>
__global__ void __launch_bounds__(kCols *kSlices)
    gemm_generic_kernel(const uint16_t *__restrict__ a, const int32_t *__restrict__ b_q,
                        const uint16_t *__restrict__ scales, const int32_t *__restrict__ qzeros,
                        int G, int zp_bias, const uint16_t *__restrict__ bias,
                        uint16_t *__restrict__ out, int64_t M, int64_t K, int64_t N) {
  using T = typename DT::T;
  __shared__ float red[kSlices][kCols * 8];

  const int tx = threadIdx.x % kCols;
  const int ts = threadIdx.x / kCols;
  const int64_t nw = N / 8;
  const int64_t c = int64_t(blockIdx.y) * kCols + tx;
  const int64_t m0 = int64_t(blockIdx.x) * kRows;
  const int rows = static_cast<int>(M - m0 < kRows ? M - m0 : kRows);
  const bool col_ok = c < nw;

  float acc[kRows][8];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[r][j] = 0.f;

  if (col_ok) {
    int64_t g_cur = -1;
    float s[8];
    int zp[8];
    for (int64_t k = ts; k < K; k += kSlices) {
      const int64_t g = k / G;
      if (g != g_cur) {
        g_cur = g;
        const uint32_t z = qzeros ? static_cast<uint32_t>(qzeros[g * nw + c]) : 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          s[j] = bits_to_float(scales[g * N + c * 8 + j], DT::kBF16);
          zp[j] = qzeros ? int((z >> (4 * j)) & 0xF) : zp_bias;
        }
      }
      const uint32_t w = static_cast<uint32_t>(b_q[k * nw + c]);
      float wv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int q = (w >> (4 * j)) & 0xF;
        wv[j] = DT::to_float(DT::from_float_rn(float(q - zp[j]) * s[j]));  // exact product, one rounding
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (r < rows) {
          const float av = bits_to_float(a[(m0 + r) * K + k], DT::kBF16);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[r][j] = fmaf(av, wv[j], acc[r][j]);
        }
      }
    }
  }

  // Sum the K slices in a fixed order, one row of A at a time (unrolled: acc stays in registers;
  // `rows` is uniform across the CTA, so the barriers below are reached by every thread).
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (r >= rows) break;
#pragma unroll
    for (int j = 0; j < 8; ++j) red[ts][tx * 8 + j] = acc[r][j];
    __syncthreads();
    {
      const int o = threadIdx.x;  // 256 outputs = 32 words x 8 columns
      const int64_t n = int64_t(blockIdx.y) * kCols * 8 + o;
      if (n < N) {
        float v = 0.f;
#pragma unroll
        for (int t = 0; t < kSlices; ++t) v += red[t][o];
        if (bias) v += bits_to_float(bias[n], DT::kBF16);
        const T y = DT::from_float_rn(v);
        out[(m0 + r) * N + n] = *reinterpret_cast<const uint16_t *>(&y);
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_gemm_generic(const GemmArgs &g) {
  const int64_t nw = g.N / 8;
  // x: row tiles of A (up to 2^31 - 1), y: column tiles (up to 65535, i.e. N <= 16.7M)
  dim3 grid(static_cast<unsigned>((g.M + kRows - 1) / kRows),
            static_cast<unsigned>((nw + kCols - 1) / kCols));
  const auto *a = static_cast<const uint16_t *>(g.a);
  const auto *sc = static_cast<const uint16_t *>(g.scales);
  const auto *bi = static_cast<const uint16_t *>(g.bias);
  auto *o = static_cast<uint16_t *>(g.out);
  if (g.dtype == W4A16_BF16)
    gemm_generic_kernel<BF16><<<grid, kCols * kSlices, 0, g.stream>>>(
        a, g.b_q, sc, g.qzeros, g.group_size, g.zp_bias, bi, o, g.M, g.K, g.N);
  else
    gemm_generic_kernel<F16><<<grid, kCols * kSlices, 0, g.stream>>>(
        a, g.b_q, sc, g.qzeros, g.group_size, g.zp_bias, bi, o, g.M, g.K, g.N);
  note_launch();
  return cudaGetLastError();
}

}  // namespace w4a16

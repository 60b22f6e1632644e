// Layout kernels: pack / unpack of 4-bit values eight per int32 along the last dimension, the
// K-packed -> N-packed repack, this library's prepacked (kernel-native) weight layout, and the
// materialised dequantisation W[k, n] = RNE_dtype((q - zp) * s).
//
// Packing: nibble j (bits 4j..4j+3) of word c holds column 8c+j - the plain reading of "eight values
// packed along N" (PR #51453 report, implementation breakdown: N = b_q.shape[1] * 8).
// Dequantisation: (raw - zero_point) * scale with group rows along K (PR #40977 report, key source
// snippets, test reference).
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t items) {
  int64_t blocks = (items + kThreads - 1) / kThreads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;  // grid-stride loops cover the rest
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

__global__ void pack_kernel(const uint8_t *__restrict__ q, int32_t *__restrict__ packed,
                            int64_t words) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < words;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint8_t *src = q + i * 8;  // word i covers bytes [8i, 8i+8) of the row-major [rows, n]
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) w |= uint32_t(src[j] & 0xF) << (4 * j);
    packed[i] = static_cast<int32_t>(w);
  }
}

__global__ void unpack_kernel(const int32_t *__restrict__ packed, uint8_t *__restrict__ q,
                              int64_t words) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < words;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint32_t w = static_cast<uint32_t>(packed[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) q[i * 8 + j] = static_cast<uint8_t>((w >> (4 * j)) & 0xF);
  }
}

// [N, K/8] -> [K, N/8]: one thread per 8x8 block of 4-bit values; it reads the eight K-packed words
// of columns 8bn..8bn+7 (word c: rows 8c..8c+7) and writes the eight N-packed words of rows
// 8c..8c+7 (word bn: columns 8bn..8bn+7), consecutive threads writing consecutive words.
__global__ void repack_k_to_n_kernel(const int32_t *__restrict__ kp, int32_t *__restrict__ np, int64_t K,
                                     int64_t N) {
  const int64_t kw = K / 8, nw = N / 8;
  const int64_t blocks = kw * nw;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < blocks;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t c = i / nw, bn = i - c * nw;
    uint32_t in[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) in[t] = static_cast<uint32_t>(kp[(8 * bn + t) * kw + c]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) w |= ((in[t] >> (4 * j)) & 0xFu) << (4 * t);
      np[(8 * c + j) * nw + bn] = static_cast<int32_t>(w);
    }
  }
}

// Prepacked layout: one thread per destination word. Destination word i is position `pos` of row r
// of the 64 x 32-word block kb of column tile t (blocks tile-major, 2048 words each); it holds word
// w = 4 * ((pos / 4) ^ (r % 8)) + pos % 4 of the tile's row, i.e. b_q[64 kb + r][32 t + w], or zero
// past K or N/8.
__global__ void prepack_kernel(const int32_t *__restrict__ b_q, int32_t *__restrict__ b_pp, int64_t K, int64_t nw,
                               int64_t kbs, int64_t total) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i & 31);
    const int r = static_cast<int>((i >> 5) & 63);
    const int64_t blk = i >> 11;  // (t, kb)
    const int64_t t = blk / kbs, kb = blk - t * kbs;
    const int w = 4 * ((pos >> 2) ^ (r & 7)) + (pos & 3);
    const int64_t k = kb * 64 + r, c = t * 32 + w;
    b_pp[i] = (k < K && c < nw) ? b_q[k * nw + c] : 0;
  }
}

template <class DT>
__global__ void dequant_kernel(const int32_t *__restrict__ b_q, const uint16_t *__restrict__ scales,
                               const int32_t *__restrict__ qzeros, int64_t K, int64_t N, int G,
                               int zp_bias, uint16_t *__restrict__ w_out) {
  using T = typename DT::T;
  const int64_t nw = N / 8;
  const int64_t words = K * nw;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < words;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t k = i / nw, c = i - k * nw;
    const int64_t g = k / G;
    const uint32_t w = static_cast<uint32_t>(b_q[i]);
    const uint32_t z = qzeros ? static_cast<uint32_t>(qzeros[g * nw + c]) : 0u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = (w >> (4 * j)) & 0xF;
      const int zp = qzeros ? int((z >> (4 * j)) & 0xF) : zp_bias;
      const float s = bits_to_float(scales[g * N + c * 8 + j], DT::kBF16);
      // (q - zp) is an integer in [-15, 15]: the fp32 product is exact, so this is one rounding.
      const T v = DT::from_float_rn(float(q - zp) * s);
      w_out[k * N + c * 8 + j] = *reinterpret_cast<const uint16_t *>(&v);
    }
  }
}

}  // namespace

cudaError_t launch_pack(const uint8_t *q, int32_t *packed, int64_t rows, int64_t n, cudaStream_t s) {
  const int64_t words = rows * (n / 8);
  if (words == 0) return cudaSuccess;
  pack_kernel<<<grid_for(words), kThreads, 0, s>>>(q, packed, words);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_unpack(const int32_t *packed, uint8_t *q, int64_t rows, int64_t n, cudaStream_t s) {
  const int64_t words = rows * (n / 8);
  if (words == 0) return cudaSuccess;
  unpack_kernel<<<grid_for(words), kThreads, 0, s>>>(packed, q, words);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_repack_k_to_n(const int32_t *k_packed, int32_t *b_q, int64_t k, int64_t n, cudaStream_t s) {
  const int64_t blocks = (k / 8) * (n / 8);
  if (blocks == 0) return cudaSuccess;
  repack_k_to_n_kernel<<<grid_for(blocks), kThreads, 0, s>>>(k_packed, b_q, k, n);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_prepack(const int32_t *b_q, int32_t *b_pp, int64_t k, int64_t n, cudaStream_t s) {
  const int64_t nw = n / 8, kbs = (k + 63) / 64, tiles = (nw + 31) / 32;
  const int64_t total = tiles * kbs * 2048;
  if (total == 0) return cudaSuccess;
  prepack_kernel<<<grid_for(total), kThreads, 0, s>>>(b_q, b_pp, k, nw, kbs, total);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_dequant(const int32_t *b_q, const void *scales, const int32_t *qzeros, int64_t k,
                           int64_t n, int group_size, int zp_bias, int dtype, void *w_out,
                           cudaStream_t s) {
  const int64_t words = k * (n / 8);
  if (words == 0) return cudaSuccess;
  const auto *sc = static_cast<const uint16_t *>(scales);
  auto *wo = static_cast<uint16_t *>(w_out);
  if (dtype == W4A16_BF16)
    dequant_kernel<BF16><<<grid_for(words), kThreads, 0, s>>>(b_q, sc, qzeros, k, n, group_size,
                                                               zp_bias, wo);
  else
    dequant_kernel<F16><<<grid_for(words), kThreads, 0, s>>>(b_q, sc, qzeros, k, n, group_size,
                                                              zp_bias, wo);
  note_launch();
  return cudaGetLastError();
}

}  // namespace w4a16

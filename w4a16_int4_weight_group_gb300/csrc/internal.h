// Host-side interfaces between the translation units of libw4a16.so (not part of the C ABI).
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/w4a16.h"

namespace w4a16 {

struct GemmArgs {
  const void *a;
  const int32_t *b_q;
  const void *scales;
  const int32_t *qzeros;  // may be null
  int group_size;
  int zp_bias;
  const void *bias;  // may be null
  void *out;
  int64_t M, K, N;
  int dtype;  // w4a16_dtype
  cudaStream_t stream;
  void *workspace = nullptr;     // optional caller-owned scratch (w4a16_gemm_ws)
  size_t workspace_bytes = 0;
  // Weights in the prepacked layout (w4a16_prepack) instead of b_q: 64-row x 32-word blocks, tile-
  // major, each 8 KB contiguous and already in the shared-memory order the kernels read.
  const int32_t *b_pp = nullptr;
};

struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;  // bytes of dynamic shared memory a CTA may opt into
  int cc_major, cc_minor;
};

// Cached per-device properties of the current device (queried once per device).
cudaError_t current_device_info(DeviceInfo *info);

// The dispatcher's plan for a call (kept per shape, dtype, alignment, workspace offer and device).
void cached_plan(const GemmArgs &g, const DeviceInfo &dev, bool workspace, w4a16_plan_t *plan);

// Records one kernel launch in the process-wide counter.
void note_launch();

// 2-D tiled TMA descriptor over a row-major [outer, inner] tensor (inner contiguous), box
// [box_outer, box_inner], zero fill outside the tensor. elem_bytes is 2 or 4. Returns false when the
// driver rejects it or the encoder is unavailable.
bool tma_encode_2d(CUtensorMap *map, int elem_bytes, const void *ptr, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle_128b);
bool tma_available();

cudaError_t launch_pack(const uint8_t *q, int32_t *packed, int64_t rows, int64_t n, cudaStream_t s);
cudaError_t launch_unpack(const int32_t *packed, uint8_t *q, int64_t rows, int64_t n, cudaStream_t s);
cudaError_t launch_repack_k_to_n(const int32_t *k_packed, int32_t *b_q, int64_t k, int64_t n, cudaStream_t s);
cudaError_t launch_prepack(const int32_t *b_q, int32_t *b_pp, int64_t k, int64_t n, cudaStream_t s);
// Bytes of the prepacked layout of a [k, n] weight matrix (K and N padded to 64 and 256).
inline size_t prepack_bytes(int64_t k, int64_t n) {
  return static_cast<size_t>((n + 255) / 256) * static_cast<size_t>((k + 63) / 64) * 8192u;
}
cudaError_t launch_dequant(const int32_t *b_q, const void *scales, const int32_t *qzeros, int64_t k,
                           int64_t n, int group_size, int zp_bias, int dtype, void *w_out,
                           cudaStream_t s);

cudaError_t launch_gemm_generic(const GemmArgs &g);

// TMA descriptors of a layer's weights (packed weights, scales, zero points), encoded once by a
// prepared layer and reused by its calls. `key` names the box shape they were encoded for (decode:
// K blocks per stage; prefill: 0).
struct WeightMaps {
  CUtensorMap tP, tS, tZ;
  int key;
};

// Decode path (M <= 32): plan fields m_tile and k_split are honoured.
bool decode_supported(const GemmArgs &g);
// query_device: use the runtime's occupancy queries (needs a device); otherwise assume 2 CTAs per SM.
void decode_make_plan(int64_t M, int64_t K, int64_t N, int group_size, int num_sms, bool query_device,
                      w4a16_plan_t *p);
// Weight descriptors for a decode plan; false when the driver rejects them.
bool decode_weight_maps(const GemmArgs &g, const w4a16_plan_t &p, WeightMaps *wm);
// wm: weight descriptors encoded for this plan, or null (encoded per call).
cudaError_t launch_gemm_decode(const GemmArgs &g, const w4a16_plan_t &p, const WeightMaps *wm = nullptr);
// Override of the decode plan's consumer groups, split-K factor and stage size (0: automatic).
void decode_set_override(int ncg, int c, int sb);
// Changes whenever a debug setting that alters plans changes (cached plans are dropped then).
uint64_t plan_epoch();
cudaError_t decode_take_device_error(uint32_t *err);
cudaError_t decode_set_wait_limit_ns(uint64_t ns);
cudaError_t decode_set_stall(bool on);

// Prefill path (tcgen05).
bool prefill_supported(const GemmArgs &g);
// workspace: a scratch buffer will be available (stream-K may be chosen).
void prefill_make_plan(int64_t M, int64_t K, int64_t N, int group_size, int num_sms, bool workspace,
                       bool query_device, w4a16_plan_t *p);
size_t prefill_workspace_bytes(int64_t M, int64_t K, int64_t N, int group_size, int num_sms);
// Whole waves of tiles a stream-K plan over `grid` CTAs runs data-parallel before the shared units.
int prefill_dp_waves(int64_t tiles, int64_t nk, int64_t grid);
// Workspace bytes a prefill plan needs (0 unless it is stream-K).
size_t prefill_plan_workspace_bytes(const w4a16_plan_t &plan);
// Device address and size of the library's static scratch array on the current device (looked up
// once per device).
cudaError_t prefill_static_scratch(void **ptr, size_t *bytes);
bool prefill_weight_maps(const GemmArgs &g, WeightMaps *wm);
cudaError_t launch_gemm_prefill(const GemmArgs &g, const w4a16_plan_t &p, const WeightMaps *wm = nullptr);
// Reads and clears the device error word of the prefill kernels on the current device.
cudaError_t prefill_take_device_error(uint32_t *err);
cudaError_t prefill_set_wait_limit_ns(uint64_t ns);
cudaError_t prefill_set_stall(bool on);

}  // namespace w4a16

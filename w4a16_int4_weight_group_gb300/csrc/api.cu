// C ABI of libw4a16.so: argument validation, the runtime dispatcher and the entry points.
//
// Validation mirrors TritonW4A16LinearKernel.can_implement (PR #43731 report, key source snippets):
// fp16/bf16 activations only, N % 8 == 0 ("8 int4 values packed per int32"), no activation
// reordering, group size in the supported list or equal to K. The tile / split-K / cluster choice is
// made on every call from the runtime M, K, N, G and the device, inside the library: the PR #51453
// report (motivation) traces a decode throughput regression to a compiler freezing the Python tile
// selection of the prefill shape into decode calls.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "internal.h"

namespace w4a16 {
namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};

w4a16_status fail(w4a16_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

w4a16_status ok() {
  g_last_error.clear();
  return W4A16_OK;
}

w4a16_status cuda_fail(cudaError_t e, const char *what) {
  return fail(W4A16_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range range(const void *p, int64_t bytes) {
  const auto lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + static_cast<uintptr_t>(bytes)};
}
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

constexpr int64_t kMaxDim = int64_t(1) << 31;
constexpr int64_t kMaxN = int64_t(1) << 24;  // column tiles index a grid dimension of at most 65535

bool group_size_ok(int G, int64_t K) { return G == 32 || G == 64 || G == 128 || int64_t(G) == K; }

// Shared rules of w4a16_can_implement / w4a16_dequant / w4a16_gemm (host only, no device access).
w4a16_status check_config(int64_t K, int64_t N, int G, int dtype) {
  if (dtype != W4A16_F16 && dtype != W4A16_BF16)
    return fail(W4A16_ERR_UNSUPPORTED, "Only float16/bfloat16 activations are supported (dtype %d)", dtype);
  if (K <= 0 || N <= 0 || K >= kMaxDim || N > kMaxN)
    return fail(W4A16_ERR_INVALID_ARG, "K (%lld) must be in [1, 2^31) and N (%lld) in [1, 2^24]",
                (long long)K, (long long)N);
  if (N % 8 != 0)
    return fail(W4A16_ERR_INVALID_ARG,
                "Output features (%lld) must be divisible by 8 (8 int4 values packed per int32)",
                (long long)N);
  if (!group_size_ok(G, K))
    return fail(W4A16_ERR_UNSUPPORTED, "Group size %d not supported; supported: [32, 64, 128] or K (%lld)",
                G, (long long)K);
  if (K % G != 0)
    return fail(W4A16_ERR_INVALID_ARG, "K (%lld) must be a multiple of group_size (%d)", (long long)K, G);
  return W4A16_OK;
}

// A path the dispatcher is restricted to (tests and benchmarks only): set by
// w4a16_debug_force_path, initially from the environment variable W4A16_FORCE_PATH
// (generic|decode|prefill), read once. -1: no restriction; -2: not read yet.
std::atomic<int> g_forced_path{-2};
std::atomic<uint64_t> g_plan_epoch{0};
int forced_path() {
  int f = g_forced_path.load(std::memory_order_relaxed);
  if (f != -2) return f;
  const char *s = std::getenv("W4A16_FORCE_PATH");
  int v = -1;
  if (s && !std::strcmp(s, "generic")) v = W4A16_PATH_GENERIC;
  else if (s && !std::strcmp(s, "decode")) v = W4A16_PATH_DECODE;
  else if (s && !std::strcmp(s, "prefill")) v = W4A16_PATH_PREFILL;
  int expected = -2;
  g_forced_path.compare_exchange_strong(expected, v, std::memory_order_relaxed);
  return g_forced_path.load(std::memory_order_relaxed);
}

// M at and above which the tcgen05 path is preferred when it applies (the decode kernel takes up to
// 32 rows: four row tiles of 8).
constexpr int64_t kPrefillMinM = 33;

// `tma` tells whether the driver's tensor-map encoder is available (the TMA-fed paths need it).
void choose_plan(const GemmArgs &g, int num_sms, bool tma, bool query_device, bool workspace, w4a16_plan_t *p) {
  std::memset(p, 0, sizeof(*p));
  if (g.M == 0) {
    p->path = W4A16_PATH_NONE;
    return;
  }
  const bool dec = tma && decode_supported(g);
  const bool pre = tma && prefill_supported(g);
  const int force = forced_path();
  int path;
  if (force == W4A16_PATH_GENERIC || (!dec && !pre)) {
    path = W4A16_PATH_GENERIC;
  } else if (force == W4A16_PATH_DECODE && dec) {
    path = W4A16_PATH_DECODE;
  } else if (force == W4A16_PATH_PREFILL && pre) {
    path = W4A16_PATH_PREFILL;
  } else if (pre && (g.M >= kPrefillMinM || !dec)) {
    path = W4A16_PATH_PREFILL;
  } else if (dec) {
    path = W4A16_PATH_DECODE;
  } else {
    path = W4A16_PATH_GENERIC;
  }
  if (path == W4A16_PATH_DECODE) {
    decode_make_plan(g.M, g.K, g.N, g.group_size, num_sms, query_device, p);
  } else if (path == W4A16_PATH_PREFILL) {
    prefill_make_plan(g.M, g.K, g.N, g.group_size, num_sms, workspace, query_device, p);
  } else {
    p->path = W4A16_PATH_GENERIC;
    p->m_tile = 8;
    p->n_tile = 256;
    p->k_split = 1;
    p->warps = 8;
    p->grid = ((g.M + 7) / 8) * ((g.N / 8 + 31) / 32);
  }
}

// The dispatcher's choice depends on the shape, the dtype, whether zero points are given, which
// pointers are 16-byte aligned, whether a workspace is offered, the forced path and the device.
// Plans are kept per such key, so that a repeated shape costs one lookup on the host.
struct PlanKey {
  int64_t M, K, N;
  int G, dtype, device, force;
  uint32_t flags;
  bool operator==(const PlanKey &o) const {
    return M == o.M && K == o.K && N == o.N && G == o.G && dtype == o.dtype && device == o.device &&
           force == o.force && flags == o.flags;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey &k) const {
    uint64_t h = 1469598103934665603ull;
    auto mix = [&](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
    mix(uint64_t(k.M)); mix(uint64_t(k.K)); mix(uint64_t(k.N)); mix(uint64_t(k.G));
    mix(uint64_t(k.dtype) | (uint64_t(k.device) << 8) | (uint64_t(k.force + 8) << 24) | (uint64_t(k.flags) << 32));
    return static_cast<size_t>(h);
  }
};

uint32_t plan_flags(const GemmArgs &g, bool workspace, bool tma) {
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return (g.qzeros ? 1u : 0u) | (workspace ? 2u : 0u) | (tma ? 4u : 0u) | (a16(g.a) ? 8u : 0u) |
         (a16(g.b_q) ? 16u : 0u) | (a16(g.scales) ? 32u : 0u) | (!g.qzeros || a16(g.qzeros) ? 64u : 0u) |
         (a16(g.out) ? 128u : 0u) | (!g.bias || a16(g.bias) ? 256u : 0u);
}

}  // namespace

uint64_t plan_epoch() { return g_plan_epoch.load(std::memory_order_relaxed); }

void cached_plan(const GemmArgs &g, const DeviceInfo &dev, bool workspace, w4a16_plan_t *plan) {
  static std::mutex mu;
  static std::unordered_map<PlanKey, w4a16_plan_t, PlanKeyHash> plans;
  static uint64_t epoch = 0;
  const bool tma = tma_available();
  const PlanKey key{g.M, g.K, g.N, g.group_size, g.dtype, dev.device, forced_path(), plan_flags(g, workspace, tma)};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (epoch != plan_epoch()) {  // a debug setting changed: plans made before it are stale
      plans.clear();
      epoch = plan_epoch();
    }
    auto it = plans.find(key);
    if (it != plans.end()) {
      *plan = it->second;
      return;
    }
  }
  choose_plan(g, dev.num_sms, tma, /*query_device=*/true, workspace, plan);
  std::lock_guard<std::mutex> lock(mu);
  if (plans.size() >= 4096) plans.clear();  // bounded: a workload with ever-new shapes re-plans
  plans.emplace(key, *plan);
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn tma_encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}
}  // namespace

bool tma_available() { return tma_encoder() != nullptr; }

bool tma_encode_2d(CUtensorMap *map, int elem_bytes, const void *ptr, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle_128b) {
  // The descriptor is a pure function of these arguments, and the calls of a model step encode the
  // same activation and output views step after step: each thread keeps its last eight encodings.
  struct Memo {
    CUtensorMap map;
    const void *ptr;
    uint64_t inner, outer, row_bytes;
    uint32_t box_inner, box_outer;
    int elem_bytes;
    bool swizzle, valid;
  };
  thread_local Memo memo[8];
  thread_local unsigned memo_next = 0;
  for (const Memo &m : memo) {
    if (m.valid && m.ptr == ptr && m.inner == inner && m.outer == outer && m.row_bytes == row_bytes &&
        m.box_inner == box_inner && m.box_outer == box_outer && m.elem_bytes == elem_bytes &&
        m.swizzle == swizzle_128b) {
      *map = m.map;
      return true;
    }
  }
  const EncodeFn enc = tma_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  if (enc(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Memo &m = memo[memo_next++ & 7u];
  m = Memo{*map, ptr, inner, outer, row_bytes, box_inner, box_outer, elem_bytes, swizzle_128b, true};
  return true;
}

cudaError_t current_device_info(DeviceInfo *info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && have[dev]) {
    *info = cache[dev];
    return cudaSuccess;
  }
  DeviceInfo d{};
  d.device = dev;
  if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
      cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    cache[dev] = d;
    have[dev] = true;
  }
  *info = d;
  return cudaSuccess;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

const char *w4a16_version(void) { return "w4a16-gb300 0.1.0 (sm_103a)"; }

const char *w4a16_last_error(void) { return g_last_error.c_str(); }

uint64_t w4a16_debug_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

w4a16_status w4a16_can_implement(int64_t k, int64_t n, int group_size, int dtype, int has_g_idx) {
  if (dtype != W4A16_F16 && dtype != W4A16_BF16)
    return fail(W4A16_ERR_UNSUPPORTED, "Only float16/bfloat16 activations are supported (dtype %d)", dtype);
  if (n > 0 && n % 8 != 0)
    return fail(W4A16_ERR_INVALID_ARG,
                "Output features (%lld) must be divisible by 8 (8 int4 values packed per int32)",
                (long long)n);
  if (has_g_idx)
    return fail(W4A16_ERR_UNSUPPORTED, "Activation reordering (g_idx) is not supported");
  const w4a16_status st = check_config(k, n, group_size, dtype);
  if (st != W4A16_OK) return st;
  return ok();
}

w4a16_status w4a16_pack(const uint8_t *q, int32_t *packed, int64_t rows, int64_t n,
                        w4a16_stream_t stream) {
  if (rows < 0 || n <= 0 || rows >= kMaxDim || n >= kMaxDim)
    return fail(W4A16_ERR_INVALID_ARG, "rows (%lld) must be >= 0 and n (%lld) > 0", (long long)rows,
                (long long)n);
  if (n % 8) return fail(W4A16_ERR_INVALID_ARG, "n (%lld) must be divisible by 8", (long long)n);
  if (rows == 0) return ok();
  if (!q || !packed) return fail(W4A16_ERR_INVALID_ARG, "q and packed must not be NULL");
  if (!aligned(packed, 4)) return fail(W4A16_ERR_MISALIGNED, "packed must be 4-byte aligned");
  if (overlaps(range(q, rows * n), range(packed, rows * n / 2)))
    return fail(W4A16_ERR_INVALID_ARG, "q and packed overlap");
  const cudaError_t e = launch_pack(q, packed, rows, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_pack launch");
  return ok();
}

w4a16_status w4a16_unpack(const int32_t *packed, uint8_t *q, int64_t rows, int64_t n,
                          w4a16_stream_t stream) {
  if (rows < 0 || n <= 0 || rows >= kMaxDim || n >= kMaxDim)
    return fail(W4A16_ERR_INVALID_ARG, "rows (%lld) must be >= 0 and n (%lld) > 0", (long long)rows,
                (long long)n);
  if (n % 8) return fail(W4A16_ERR_INVALID_ARG, "n (%lld) must be divisible by 8", (long long)n);
  if (rows == 0) return ok();
  if (!q || !packed) return fail(W4A16_ERR_INVALID_ARG, "q and packed must not be NULL");
  if (!aligned(packed, 4)) return fail(W4A16_ERR_MISALIGNED, "packed must be 4-byte aligned");
  if (overlaps(range(q, rows * n), range(packed, rows * n / 2)))
    return fail(W4A16_ERR_INVALID_ARG, "q and packed overlap");
  const cudaError_t e = launch_unpack(packed, q, rows, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_unpack launch");
  return ok();
}

w4a16_status w4a16_repack_k_to_n(const int32_t *k_packed, int32_t *b_q, int64_t k, int64_t n,
                                 w4a16_stream_t stream) {
  if (k <= 0 || n <= 0 || k >= kMaxDim || n >= kMaxDim)
    return fail(W4A16_ERR_INVALID_ARG, "k (%lld) and n (%lld) must be > 0", (long long)k, (long long)n);
  if (k % 8 || n % 8)
    return fail(W4A16_ERR_INVALID_ARG, "k (%lld) and n (%lld) must be divisible by 8", (long long)k, (long long)n);
  if (!k_packed || !b_q) return fail(W4A16_ERR_INVALID_ARG, "k_packed and b_q must not be NULL");
  if (!aligned(k_packed, 4) || !aligned(b_q, 4)) return fail(W4A16_ERR_MISALIGNED, "k_packed and b_q must be 4-byte aligned");
  if (overlaps(range(k_packed, k * n / 2), range(b_q, k * n / 2)))
    return fail(W4A16_ERR_INVALID_ARG, "k_packed and b_q overlap");
  const cudaError_t e = launch_repack_k_to_n(k_packed, b_q, k, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_repack_k_to_n launch");
  return ok();
}

size_t w4a16_prepack_bytes(int64_t k, int64_t n) {
  if (k <= 0 || n <= 0 || k >= kMaxDim || n > kMaxN || n % 8) return 0;
  return prepack_bytes(k, n);
}

w4a16_status w4a16_prepack(const int32_t *b_q, int32_t *b_pp, int64_t k, int64_t n, w4a16_stream_t stream) {
  if (k <= 0 || n <= 0 || k >= kMaxDim || n > kMaxN)
    return fail(W4A16_ERR_INVALID_ARG, "k (%lld) and n (%lld) must be > 0", (long long)k, (long long)n);
  if (n % 8) return fail(W4A16_ERR_INVALID_ARG, "n (%lld) must be divisible by 8", (long long)n);
  if (!b_q || !b_pp) return fail(W4A16_ERR_INVALID_ARG, "b_q and b_pp must not be NULL");
  if (!aligned(b_q, 4) || !aligned(b_pp, 16))
    return fail(W4A16_ERR_MISALIGNED, "b_q must be 4-byte and b_pp 16-byte aligned");
  if (overlaps(range(b_q, k * n / 2), range(b_pp, static_cast<int64_t>(prepack_bytes(k, n)))))
    return fail(W4A16_ERR_INVALID_ARG, "b_q and b_pp overlap");
  const cudaError_t e = launch_prepack(b_q, b_pp, k, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_prepack launch");
  return ok();
}

w4a16_status w4a16_dequant(const int32_t *b_q, const void *scales, const int32_t *qzeros, int64_t k,
                           int64_t n, int group_size, int zp_bias, w4a16_dtype dtype, void *w_out,
                           w4a16_stream_t stream) {
  w4a16_status st = check_config(k, n, group_size, dtype);
  if (st != W4A16_OK) return st;
  if (!qzeros && (zp_bias < 0 || zp_bias > 15))
    return fail(W4A16_ERR_INVALID_ARG, "zp_bias (%d) must be in [0, 15]", zp_bias);
  if (!b_q || !scales || !w_out) return fail(W4A16_ERR_INVALID_ARG, "b_q, scales and w_out must not be NULL");
  if (!aligned(b_q, 4) || !aligned(scales, 2) || !aligned(w_out, 2) || (qzeros && !aligned(qzeros, 4)))
    return fail(W4A16_ERR_MISALIGNED, "tensors must be naturally aligned");
  const Range wo = range(w_out, k * n * 2);
  if (overlaps(wo, range(b_q, k * n / 2)) || overlaps(wo, range(scales, (k / group_size) * n * 2)) ||
      (qzeros && overlaps(wo, range(qzeros, (k / group_size) * n / 2))))
    return fail(W4A16_ERR_INVALID_ARG, "w_out overlaps an input");
  const cudaError_t e = launch_dequant(b_q, scales, qzeros, k, n, group_size, zp_bias, dtype, w_out,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_dequant launch");
  return ok();
}

static w4a16_status validate_gemm(const GemmArgs &g) {
  w4a16_status st = check_config(g.K, g.N, g.group_size, g.dtype);
  if (st != W4A16_OK) return st;
  if (g.M < 0 || g.M >= kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "M (%lld) must be in [0, 2^31)", (long long)g.M);
  if (!g.qzeros && (g.zp_bias < 0 || g.zp_bias > 15))
    return fail(W4A16_ERR_INVALID_ARG, "zp_bias (%d) must be in [0, 15]", g.zp_bias);
  if (g.M == 0) return W4A16_OK;
  if (!g.a || !g.b_q || !g.scales || !g.out)
    return fail(W4A16_ERR_INVALID_ARG, "a, b_q, scales and out must not be NULL");
  if (!aligned(g.a, 2) || !aligned(g.b_q, 4) || !aligned(g.scales, 2) || !aligned(g.out, 2) ||
      (g.qzeros && !aligned(g.qzeros, 4)) || (g.bias && !aligned(g.bias, 2)))
    return fail(W4A16_ERR_MISALIGNED, "tensors must be naturally aligned (2 bytes for 16-bit, 4 for int32)");
  const int64_t ng = g.K / g.group_size;
  const Range o = range(g.out, g.M * g.N * 2);
  if (overlaps(o, range(g.a, g.M * g.K * 2)) || overlaps(o, range(g.b_q, g.K * g.N / 2)) ||
      overlaps(o, range(g.scales, ng * g.N * 2)) || (g.qzeros && overlaps(o, range(g.qzeros, ng * g.N / 2))) ||
      (g.bias && overlaps(o, range(g.bias, g.N * 2))))
    return fail(W4A16_ERR_INVALID_ARG, "out overlaps an input tensor");
  return W4A16_OK;
}

static w4a16_status gemm_impl(GemmArgs &g) {
  w4a16_status st = validate_gemm(g);
  if (st != W4A16_OK) return st;
  if (g.M == 0) return ok();
  if (g.workspace && !aligned(g.workspace, 256))
    return fail(W4A16_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  w4a16_plan_t plan;
  cached_plan(g, dev, g.workspace != nullptr, &plan);
  // a stream-K plan whose workspace the caller did not provide in full falls back to whole tiles
  if (g.workspace && g.workspace_bytes < prefill_plan_workspace_bytes(plan)) cached_plan(g, dev, false, &plan);
  switch (plan.path) {
    case W4A16_PATH_DECODE: e = launch_gemm_decode(g, plan); break;
    case W4A16_PATH_PREFILL: e = launch_gemm_prefill(g, plan); break;
    default: e = launch_gemm_generic(g); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_gemm launch");
  return ok();
}

w4a16_status w4a16_gemm(const void *a, const int32_t *b_q, const void *scales, const int32_t *qzeros,
                        int group_size, int zp_bias, const void *bias, void *out, int64_t m,
                        int64_t k, int64_t n, w4a16_dtype dtype, w4a16_stream_t stream) {
  GemmArgs g{a, b_q, scales, qzeros, group_size, zp_bias, bias, out, m, k, n, static_cast<int>(dtype),
             reinterpret_cast<cudaStream_t>(stream)};
  return gemm_impl(g);
}

w4a16_status w4a16_gemm_ws(const void *a, const int32_t *b_q, const void *scales, const int32_t *qzeros,
                           int group_size, int zp_bias, const void *bias, void *out, int64_t m, int64_t k,
                           int64_t n, w4a16_dtype dtype, void *workspace, size_t workspace_bytes,
                           w4a16_stream_t stream) {
  GemmArgs g{a, b_q, scales, qzeros, group_size, zp_bias, bias, out, m, k, n, static_cast<int>(dtype),
             reinterpret_cast<cudaStream_t>(stream)};
  g.workspace = workspace;
  g.workspace_bytes = workspace ? workspace_bytes : 0;
  if (workspace) {
    const Range w = range(workspace, static_cast<int64_t>(workspace_bytes));
    const int64_t ng = (group_size > 0 && k > 0) ? k / group_size : 0;
    if (overlaps(w, range(out, m * n * 2)) || overlaps(w, range(a, m * k * 2)) ||
        overlaps(w, range(b_q, k * n / 2)) || overlaps(w, range(scales, ng * n * 2)) ||
        (qzeros && overlaps(w, range(qzeros, ng * n / 2))) || (bias && overlaps(w, range(bias, n * 2))))
      return fail(W4A16_ERR_INVALID_ARG, "workspace overlaps a tensor argument");
  }
  return gemm_impl(g);
}

w4a16_status w4a16_gemm_noalloc(const void *a, const int32_t *b_q, const void *scales,
                                const int32_t *qzeros, int group_size, int zp_bias, const void *bias,
                                void *out, int64_t m, int64_t k, int64_t n, w4a16_dtype dtype,
                                w4a16_stream_t stream) {
  GemmArgs g{a, b_q, scales, qzeros, group_size, zp_bias, bias, out, m, k, n, static_cast<int>(dtype),
             reinterpret_cast<cudaStream_t>(stream)};
  w4a16_status st = validate_gemm(g);
  if (st != W4A16_OK) return st;
  if (m == 0) return ok();
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  void *scratch = nullptr;
  size_t scratch_bytes = 0;
  e = prefill_static_scratch(&scratch, &scratch_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "static scratch address (cudaGetSymbolAddress)");
  // the plan this call will run (gemm_impl makes the same choice); only stream-K needs scratch
  w4a16_plan_t plan;
  cached_plan(g, dev, /*workspace=*/true, &plan);
  const size_t need = prefill_plan_workspace_bytes(plan);
  if (need > scratch_bytes)
    return fail(W4A16_ERR_UNSUPPORTED,
                "this call needs %zu bytes of scratch (stream-K over %d SMs); the static scratch holds %zu",
                need, dev.num_sms, scratch_bytes);
  if (need > 0) {
    // The array keeps the previous call's contents: the stream-K flags (one word per CTA at the
    // start of the scratch) must start at zero.
    e = cudaMemsetAsync(scratch, 0, static_cast<size_t>(plan.grid) * 4, g.stream);
    if (e != cudaSuccess) return cuda_fail(e, "clear static scratch flags");
  }
  g.workspace = scratch;
  g.workspace_bytes = scratch_bytes;
  return gemm_impl(g);
}

}  // extern "C"

// A prepared layer: the weights' configuration checked once, the dispatcher's plan and the weight
// descriptors kept per call shape, so that a call validates and encodes only the activations.
struct w4a16_layer_st {
  GemmArgs proto;  // weights, group size, zero points, bias, K, N, dtype
  int device = 0;
  struct Entry {
    w4a16_plan_t plan;
    WeightMaps maps;
    bool have_maps;
  };
  std::mutex mu;
  std::unordered_map<uint64_t, Entry> cache;  // key: M, plan flags, forced path
  uint64_t epoch = 0;                          // plan_epoch() the entries were made under
};

extern "C" {

static w4a16_status layer_create(const int32_t *b_q, const int32_t *b_pp, const void *scales, const int32_t *qzeros,
                                 int group_size, int zp_bias, const void *bias, int64_t k, int64_t n, w4a16_dtype dtype,
                                 w4a16_layer_t *layer) {
  if (!layer) return fail(W4A16_ERR_INVALID_ARG, "layer must not be NULL");
  *layer = nullptr;
  w4a16_status st = check_config(k, n, group_size, dtype);
  if (st != W4A16_OK) return st;
  if (!qzeros && (zp_bias < 0 || zp_bias > 15))
    return fail(W4A16_ERR_INVALID_ARG, "zp_bias (%d) must be in [0, 15]", zp_bias);
  if (!(b_q || b_pp) || !scales) return fail(W4A16_ERR_INVALID_ARG, "the weights and scales must not be NULL");
  if ((b_q && !aligned(b_q, 4)) || (b_pp && !aligned(b_pp, 16)) || !aligned(scales, 2) ||
      (qzeros && !aligned(qzeros, 4)) || (bias && !aligned(bias, 2)))
    return fail(W4A16_ERR_MISALIGNED, "tensors must be naturally aligned (2 bytes for 16-bit, 4 for int32, 16 for "
                "prepacked weights)");
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  auto *L = new (std::nothrow) w4a16_layer_st;
  if (!L) return fail(W4A16_ERR_INVALID_ARG, "out of host memory");
  L->proto = GemmArgs{nullptr, b_q, scales, qzeros, group_size, zp_bias, bias, nullptr, 0, k, n,
                      static_cast<int>(dtype), nullptr};
  L->proto.b_pp = b_pp;
  L->device = dev;
  *layer = L;
  return ok();
}

w4a16_status w4a16_layer_create(const int32_t *b_q, const void *scales, const int32_t *qzeros, int group_size,
                                int zp_bias, const void *bias, int64_t k, int64_t n, w4a16_dtype dtype,
                                w4a16_layer_t *layer) {
  if (!b_q) {
    if (layer) *layer = nullptr;
    return fail(W4A16_ERR_INVALID_ARG, "b_q and scales must not be NULL");
  }
  return layer_create(b_q, nullptr, scales, qzeros, group_size, zp_bias, bias, k, n, dtype, layer);
}

w4a16_status w4a16_layer_create_prepacked(const int32_t *b_pp, const void *scales, const int32_t *qzeros,
                                          int group_size, int zp_bias, const void *bias, int64_t k, int64_t n,
                                          w4a16_dtype dtype, w4a16_layer_t *layer) {
  if (!b_pp) {
    if (layer) *layer = nullptr;
    return fail(W4A16_ERR_INVALID_ARG, "b_pp and scales must not be NULL");
  }
  return layer_create(nullptr, b_pp, scales, qzeros, group_size, zp_bias, bias, k, n, dtype, layer);
}

w4a16_status w4a16_layer_destroy(w4a16_layer_t layer) {
  delete layer;
  return ok();
}

size_t w4a16_layer_workspace_size(w4a16_layer_t layer, int64_t m) {
  if (!layer) return 0;
  return w4a16_gemm_workspace_size(m, layer->proto.K, layer->proto.N, layer->proto.group_size, layer->proto.dtype);
}

w4a16_status w4a16_layer_gemm(w4a16_layer_t layer, const void *a, void *out, int64_t m, void *workspace,
                              size_t workspace_bytes, w4a16_stream_t stream) {
  if (!layer) return fail(W4A16_ERR_INVALID_ARG, "layer must not be NULL");
  GemmArgs g = layer->proto;
  g.a = a;
  g.out = out;
  g.M = m;
  g.stream = reinterpret_cast<cudaStream_t>(stream);
  g.workspace = workspace;
  g.workspace_bytes = workspace ? workspace_bytes : 0;
  if (m < 0 || m >= kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "M (%lld) must be in [0, 2^31)", (long long)m);
  if (m == 0) return ok();
  if (!a || !out) return fail(W4A16_ERR_INVALID_ARG, "a and out must not be NULL");
  if (!aligned(a, 2) || !aligned(out, 2)) return fail(W4A16_ERR_MISALIGNED, "a and out must be 2-byte aligned");
  if (workspace && !aligned(workspace, 256)) return fail(W4A16_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  const int64_t ng = g.K / g.group_size;
  const Range o = range(out, m * g.N * 2);
  const Range wt = g.b_pp ? range(g.b_pp, static_cast<int64_t>(prepack_bytes(g.K, g.N))) : range(g.b_q, g.K * g.N / 2);
  if (overlaps(o, range(a, m * g.K * 2)) || overlaps(o, wt) ||
      overlaps(o, range(g.scales, ng * g.N * 2)) || (g.qzeros && overlaps(o, range(g.qzeros, ng * g.N / 2))) ||
      (g.bias && overlaps(o, range(g.bias, g.N * 2))))
    return fail(W4A16_ERR_INVALID_ARG, "out overlaps an input tensor");
  if (workspace) {
    const Range w = range(workspace, static_cast<int64_t>(workspace_bytes));
    if (overlaps(w, o) || overlaps(w, range(a, m * g.K * 2)) || overlaps(w, wt) ||
        overlaps(w, range(g.scales, ng * g.N * 2)) || (g.qzeros && overlaps(w, range(g.qzeros, ng * g.N / 2))) ||
        (g.bias && overlaps(w, range(g.bias, g.N * 2))))
      return fail(W4A16_ERR_INVALID_ARG, "workspace overlaps a tensor argument");
  }
  DeviceInfo dev;
  cudaError_t e = current_device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  if (dev.device != layer->device)
    return fail(W4A16_ERR_INVALID_ARG, "the layer was prepared on device %d, the current device is %d", layer->device,
                dev.device);
  const bool tma = tma_available();
  const int force = forced_path();
  auto entry_for = [&](bool ws) -> w4a16_layer_st::Entry {
    const uint64_t key = (uint64_t(m) << 20) | (uint64_t(plan_flags(g, ws, tma)) << 4) | uint64_t(force + 2);
    {
      std::lock_guard<std::mutex> lock(layer->mu);
      if (layer->epoch != plan_epoch()) {
        layer->cache.clear();
        layer->epoch = plan_epoch();
      }
      auto it = layer->cache.find(key);
      if (it != layer->cache.end()) return it->second;
    }
    w4a16_layer_st::Entry en{};
    cached_plan(g, dev, ws, &en.plan);
    if (en.plan.path == W4A16_PATH_DECODE) en.have_maps = decode_weight_maps(g, en.plan, &en.maps);
    else if (en.plan.path == W4A16_PATH_PREFILL) en.have_maps = prefill_weight_maps(g, &en.maps);
    std::lock_guard<std::mutex> lock(layer->mu);
    if (layer->cache.size() >= 1024) layer->cache.clear();
    layer->cache.emplace(key, en);
    return en;
  };
  w4a16_layer_st::Entry en = entry_for(workspace != nullptr);
  // a stream-K plan whose workspace the caller did not provide in full falls back to whole tiles
  if (workspace && workspace_bytes < prefill_plan_workspace_bytes(en.plan)) en = entry_for(false);
  const WeightMaps *wm = en.have_maps ? &en.maps : nullptr;
  if (g.b_pp && en.plan.path != W4A16_PATH_DECODE && en.plan.path != W4A16_PATH_PREFILL)
    return fail(W4A16_ERR_UNSUPPORTED, "prepacked weights are read by the TMA-fed kernels only: a and out must be "
                "16-byte aligned, N %% 32 == 0 and K %% 8 == 0 (and no forced generic path)");
  switch (en.plan.path) {
    case W4A16_PATH_DECODE: e = launch_gemm_decode(g, en.plan, wm); break;
    case W4A16_PATH_PREFILL: e = launch_gemm_prefill(g, en.plan, wm); break;
    default: e = launch_gemm_generic(g); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_layer_gemm launch");
  return ok();
}

size_t w4a16_gemm_workspace_size(int64_t m, int64_t k, int64_t n, int group_size, int dtype) {
  if (check_config(k, n, group_size, dtype) != W4A16_OK || m <= 0 || m >= kMaxDim) return 0;
  DeviceInfo dev;
  if (current_device_info(&dev) != cudaSuccess) return 0;
  // the dispatcher's own choice (16-byte aligned tensors assumed): decode shapes need none
  static const int32_t kAlignedWord[4] = {0, 0, 0, 0};
  const void *p16 = reinterpret_cast<const void *>((reinterpret_cast<uintptr_t>(kAlignedWord) + 15) & ~uintptr_t(15));
  GemmArgs g{p16, static_cast<const int32_t *>(p16), p16, nullptr, group_size, 8, nullptr, const_cast<void *>(p16),
             m, k, n, dtype, nullptr};
  w4a16_plan_t plan;
  choose_plan(g, dev.num_sms, /*tma=*/true, /*query_device=*/true, /*workspace=*/true, &plan);
  return prefill_plan_workspace_bytes(plan);
}

w4a16_status w4a16_plan(int64_t m, int64_t k, int64_t n, int group_size, int dtype, int has_zp,
                        int num_sms, int with_workspace, w4a16_plan_t *plan) {
  if (!plan) return fail(W4A16_ERR_INVALID_ARG, "plan must not be NULL");
  w4a16_status st = check_config(k, n, group_size, dtype);
  if (st != W4A16_OK) return st;
  if (m < 0 || m >= kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "M (%lld) must be in [0, 2^31)", (long long)m);
  const bool query_device = num_sms <= 0;
  if (num_sms <= 0) {
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    num_sms = dev.num_sms;
  }
  // Pointers are assumed 16-byte aligned: any 16-byte aligned address stands in for them.
  static const int32_t kAlignedWord[4] = {0, 0, 0, 0};
  const void *p16 = reinterpret_cast<const void *>(
      (reinterpret_cast<uintptr_t>(kAlignedWord) + 15) & ~uintptr_t(15));
  GemmArgs g{p16, static_cast<const int32_t *>(p16), p16, has_zp ? static_cast<const int32_t *>(p16) : nullptr,
             group_size, 8, nullptr, nullptr, m, k, n, dtype, nullptr};
  // a host-only query: assume a GPU driver; use the device's occupancy only when it was asked for
  choose_plan(g, num_sms, /*tma=*/true, query_device, with_workspace != 0, plan);
  return ok();
}

int w4a16_debug_selected_path(int64_t m, int64_t k, int64_t n, int group_size) {
  w4a16_plan_t p;
  if (w4a16_plan(m, k, n, group_size, W4A16_F16, 0, 0, 0, &p) != W4A16_OK) return -1;
  return p.path;
}

w4a16_status w4a16_get_device_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "synchronise");
  uint32_t err = 0, err2 = 0;
  e = prefill_take_device_error(&err);
  if (e == cudaSuccess) e = decode_take_device_error(&err2);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  err |= err2;
  if (err) return fail(W4A16_ERR_TIMEOUT, "a bounded device-side wait gave up (code 0x%x)", err);
  return ok();
}

w4a16_status w4a16_debug_force_path(int path) {
  if (path != -1 && path != W4A16_PATH_GENERIC && path != W4A16_PATH_DECODE && path != W4A16_PATH_PREFILL)
    return fail(W4A16_ERR_INVALID_ARG, "path %d is not -1, W4A16_PATH_GENERIC, _DECODE or _PREFILL", path);
  g_forced_path.store(path, std::memory_order_relaxed);
  g_plan_epoch.fetch_add(1, std::memory_order_relaxed);
  return ok();
}

w4a16_status w4a16_debug_decode_override(int consumer_groups, int k_split, int k_blocks_per_stage) {
  if (consumer_groups < 0 || consumer_groups > 2 || k_split < 0 || k_split > 16 ||
      (k_blocks_per_stage != 0 && k_blocks_per_stage != 1 && k_blocks_per_stage != 2 && k_blocks_per_stage != 4))
    return fail(W4A16_ERR_INVALID_ARG, "override out of range: consumer_groups in 0..2, k_split in 0..16, "
                "k_blocks_per_stage in {0, 1, 2, 4}");
  decode_set_override(consumer_groups, k_split, k_blocks_per_stage);
  g_plan_epoch.fetch_add(1, std::memory_order_relaxed);
  return ok();
}

w4a16_status w4a16_debug_set_wait_limit_ns(uint64_t ns) {
  cudaError_t e = prefill_set_wait_limit_ns(ns);
  if (e == cudaSuccess) e = decode_set_wait_limit_ns(ns);
  if (e != cudaSuccess) return cuda_fail(e, "set wait limit");
  return ok();
}

w4a16_status w4a16_debug_inject_stall(int on) {
  cudaError_t e = prefill_set_stall(on != 0);
  if (e == cudaSuccess) e = decode_set_stall(on != 0);
  if (e != cudaSuccess) return cuda_fail(e, "set stall hook");
  return ok();
}

}  // extern "C"

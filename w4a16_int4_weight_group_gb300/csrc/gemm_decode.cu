// Decode / skinny path of the W4A16 product (small M): a split-K GEMM that streams the packed
// weights once from HBM, dequantises them in registers and multiplies on the tensor cores.
//
// Where the ideas come from (PR #40977 report, implementation breakdown item 3 - a split-K skinny
// decode kernel with magic-number int4 -> half dequantisation and a cross-lane reduction; PR #51453
// report, review highlights - split-K requested because small-M decode leaves the GPU idle), and what
// this kernel does on sm_103a instead:
//
//  * Work split. A CTA owns 64*V output columns (V packed words per lane per row) and 8*J rows of A.
//    Its W warps split the CTA's K range into contiguous pieces; C CTAs of one thread-block cluster
//    split K further. Partial sums are added in shared memory (warps) and through distributed shared
//    memory (cluster ranks) in a fixed order, so results are deterministic and no global scratch
//    memory is needed.
//  * Streaming. Each warp owns a ring of R shared-memory stages. One stage is one k-step of 16 rows:
//    16 x 32V bytes of packed weights, the matching 16 columns of A (rows past M zero-filled), and at
//    group starts the scale row (and zero-point words). All of it arrives by 16-byte cp.async
//    (coalesced, L2-only), R-1 stages ahead of the math, so no registers hold data in flight.
//    The weight stage layout is XOR-swizzled so that the fragment reads below are bank-conflict free.
//  * Dequantisation (magic numbers, one rounding). For two rows k, k+1 of one word column, one byte
//    permute interleaves their nibbles so that a single LOP3 places nibble j of both rows into the
//    low mantissa bits of two fp16 (exponent of 1024, or 64 for the high nibble of a byte) or bf16
//    (exponent of 128) values: the packed pair is then exactly (base+q_k, base+q_k+1). Subtracting
//    (base+zp) is exact and gives the integers q - zp; one packed multiply by the scale rounds once,
//    giving exactly RNE((q - zp) * s), the values w4a16_dequant writes.
//  * Multiply. mma.sync m16n8k16 with the weights as the 16-row operand (16 output columns) and the
//    activations as the 8-column operand (8 rows of A): the pages' M <= 8 decode batch fills the
//    n=8 side. The k order inside an MMA is a free permutation; it is chosen so that each lane's
//    k values are 4 consecutive rows (one 8-byte activation load) and each register pair is a row
//    pair (k, k+1) of one output column.
//  * Epilogue. Bias is added in fp32, the sum is rounded once to the activation dtype
//    (PR #40977 report, key source snippets, test reference).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kRing = 6;    // stages per warp

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
constexpr int kWarps = 8;   // warps per CTA

template <int V, int J, bool HAS_ZP>
struct DecodeLayout {
  static constexpr int kWN = 64 * V;                   // output columns per CTA
  static constexpr int kMT = 8 * J;                    // rows of A per CTA
  static constexpr int kWBytes = 16 * 32 * V;          // 16 rows x 8V words
  static constexpr int kABytes = kMT * 32;             // kMT rows x 16 halves
  static constexpr int kSBytes = kWN * 2;              // one scale row
  static constexpr int kZBytes = HAS_ZP ? kWN / 2 : 0; // one zero-point row (8V words)
  static constexpr int kA = kWBytes;
  static constexpr int kS = kA + kABytes;
  static constexpr int kZ = kS + kSBytes;
  static constexpr int kStage = kZ + kZBytes;
  static constexpr int kWarpRing = kStage * kRing;
  static constexpr int kRingBytes = kWarpRing * kWarps;
  static constexpr int kRedBytes = kWarps * kMT * kWN * 4;
  static constexpr int kSmem = kRingBytes > kRedBytes ? kRingBytes : kRedBytes;
  static_assert(kStage % 16 == 0, "stage must keep 16-byte alignment");
};

// Byte offset of 16-byte chunk c of weight row `row` (0..15) inside a stage. Rows are 32V bytes;
// 4/V rows share a 128-byte line, and chunk positions are XOR-swizzled by bits 2..3 of the row.
template <int V>
__device__ __forceinline__ uint32_t w_chunk_offset(int row, int c) {
  constexpr int kRowsPerLine = 4 / V;
  const int line = row / kRowsPerLine;
  const int pos = (((row % kRowsPerLine) * (2 * V)) + c) ^ (2 * ((row >> 2) & 3));
  return static_cast<uint32_t>(line * 128 + pos * 16);
}

struct DecodeParams {
  const uint16_t *a;
  const int32_t *b_q;
  const uint16_t *scales;
  const int32_t *qzeros;
  const uint16_t *bias;
  uint16_t *out;
  int64_t M, K, N;
  int G;
  int zp_bias;
  int k_split;        // C: CTAs per cluster along K
  int ksteps_per_cta; // k-steps (16 rows) per cluster rank
};

template <class DT, int V, int J, bool HAS_ZP>
__global__ void __launch_bounds__(kWarps * 32, 2)
    decode_kernel(const DecodeParams p) {
  using L = DecodeLayout<V, J, HAS_ZP>;
  using T = typename DT::T;
  constexpr bool BF = DT::kBF16;
  extern __shared__ __align__(128) uint8_t smem[];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int gl = lane >> 2;   // "groupID" of the MMA fragment layouts
  const int tig = lane & 3;   // thread in group

  const int C = p.k_split;
  const int rank = static_cast<int>(blockIdx.x % C);
  const int64_t n0 = int64_t(blockIdx.x / C) * L::kWN;
  const int64_t m0 = int64_t(blockIdx.y) * L::kMT;
  const int64_t NW = p.N / 8;
  const int64_t KS = p.K / 16;

  // K range of this CTA, then of this warp (contiguous pieces).
  const int64_t c_begin = min64(KS, int64_t(rank) * p.ksteps_per_cta);
  const int64_t c_end = min64(KS, c_begin + p.ksteps_per_cta);
  const int64_t per_warp = (c_end - c_begin + kWarps - 1) / kWarps;
  const int64_t w_begin = min64(c_end, c_begin + warp * per_warp);
  const int64_t w_end = min64(c_end, w_begin + per_warp);
  const int nsteps = static_cast<int>(w_end - w_begin);

  uint8_t *ring = smem + warp * L::kWarpRing;
  const uint32_t ring_u32 = smem_u32(ring);

  // Inputs may be written by the previous kernel in the stream: wait for it before any global
  // access, then let the next kernel start its launch while this one runs.
  griddep_wait();
  griddep_launch_dependents();

  // ---- producer state: per-lane source pointers advanced by a fixed stride per k-step ----
  // steps per scale group (G is a multiple of 16) and this warp's position inside its first group
  const int spg = p.G / 16;
  const int gpos0 = static_cast<int>(w_begin % spg);
  const int64_t g_begin = w_begin / spg;
  const int32_t *wsrc[V];
  uint32_t wdst[V];
  bool wok[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int ci = lane + 32 * u;
    const int row = ci / (2 * V), c = ci % (2 * V);
    const int64_t word = n0 / 8 + 4 * c;
    wok[u] = word < NW;
    wsrc[u] = p.b_q + (w_begin * 16 + row) * NW + (wok[u] ? word : 0);
    wdst[u] = w_chunk_offset<V>(row, c);
  }
  constexpr int kAChunks = (2 * L::kMT + 31) / 32;
  const uint16_t *asrc[kAChunks];
  uint32_t adst[kAChunks];
  bool aok[kAChunks], alane[kAChunks];
#pragma unroll
  for (int u = 0; u < kAChunks; ++u) {
    const int ci = lane + 32 * u;
    const int row = ci >> 1, c = ci & 1;
    alane[u] = ci < 2 * L::kMT;
    aok[u] = alane[u] && m0 + row < p.M;
    asrc[u] = p.a + (aok[u] ? (m0 + row) * p.K + w_begin * 16 + 8 * c : 0);
    adst[u] = L::kA + row * 32 + c * 16;
  }
  const bool s_lane = lane < L::kSBytes / 16;
  const bool s_ok = s_lane && n0 + 8 * lane < p.N;
  const uint16_t *ssrc = p.scales + g_begin * p.N + (s_ok ? n0 + 8 * lane : 0);
  const bool z_lane = HAS_ZP && lane < L::kZBytes / 16;
  const bool z_ok = z_lane && n0 / 8 + 4 * lane < NW;
  const int32_t *zsrc = HAS_ZP ? p.qzeros + g_begin * NW + (z_ok ? n0 / 8 + 4 * lane : 0) : nullptr;
  int issue_i = 0, issue_slot = 0, issue_gpos = gpos0;

  // ---- producer: issue the copies of the next local step into its slot ----
  auto issue = [&]() {
    if (issue_i < nsteps) {
      const uint32_t st = ring_u32 + issue_slot * L::kStage;
#pragma unroll
      for (int u = 0; u < V; ++u) {
        cp_async_16(st + wdst[u], wsrc[u], wok[u]);
        wsrc[u] += 16 * NW;
      }
#pragma unroll
      for (int u = 0; u < kAChunks; ++u) {
        if (alane[u]) cp_async_16(st + adst[u], asrc[u], aok[u]);
        if (aok[u]) asrc[u] += 16;
      }
      if (issue_i == 0 || issue_gpos == 0) {
        if (s_lane) cp_async_16(st + L::kS + 16 * lane, ssrc, s_ok);
        if constexpr (HAS_ZP) {
          if (z_lane) cp_async_16(st + L::kZ + 16 * lane, zsrc, z_ok);
        }
      }
      if (++issue_gpos == spg) {
        issue_gpos = 0;
        ssrc += p.N;
        if constexpr (HAS_ZP) zsrc += NW;
      }
      ++issue_i;
      if (++issue_slot == kRing) issue_slot = 0;
    }
    cp_async_commit();
  };

  // ---- per-lane constant fragment addresses inside a stage ----
  uint32_t w_off[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 4 * tig + r;
    const int byte = 4 * V * gl;  // this lane's V words inside the row
    w_off[r] = w_chunk_offset<V>(row, byte / 16) + (byte % 16);
  }

  // zero-point subtrahends (base + zp) per output column, packed twice (both k rows of a pair)
  uint32_t zsub[V][8];
  uint32_t s2[V][8];
  auto make_zsub = [&](int j, uint32_t zp) -> uint32_t {
    uint32_t h;
    if constexpr (BF) h = 0x4300u | zp;               // 128 + zp
    else h = (j & 1) ? (0x5400u | (zp << 4)) : (0x6400u | zp);  // 64 + zp  /  1024 + zp
    return h | (h << 16);
  };
  if constexpr (!HAS_ZP) {
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int j = 0; j < 8; ++j) zsub[v][j] = make_zsub(j, static_cast<uint32_t>(p.zp_bias));
  }

  float acc[J][V][4][4];
#pragma unroll
  for (int jt = 0; jt < J; ++jt)
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[jt][v][q][e] = 0.f;

  // ---- software pipeline ----
#pragma unroll
  for (int s = 0; s < kRing - 1; ++s) issue();

  int slot = 0, gpos = gpos0;
  for (int i = 0; i < nsteps; ++i) {
    issue();
    cp_async_wait<kRing - 1>();
    __syncwarp();

    const uint32_t st = ring_u32 + slot * L::kStage;
    if (++slot == kRing) slot = 0;
    const bool new_group = i == 0 || gpos == 0;
    if (++gpos == spg) gpos = 0;

    if (new_group) {
      // scale row: this lane's 8V columns start at column 8*V*gl of the tile
#pragma unroll
      for (int v = 0; v < V; ++v) {
        uint32_t sp[4];
        lds128(st + L::kS + 16 * (V * gl + v), sp[0], sp[1], sp[2], sp[3]);
#pragma unroll
        for (int j = 0; j < 8; ++j) s2[v][j] = prmt(sp[j >> 1], sp[j >> 1], (j & 1) ? 0x3232 : 0x1010);
      }
      if constexpr (HAS_ZP) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const uint32_t zw = lds32(st + L::kZ + 4 * (V * gl + v));
#pragma unroll
          for (int j = 0; j < 8; ++j) zsub[v][j] = make_zsub(j, (zw >> (4 * j)) & 0xF);
        }
      }
    }

    // activation fragments (B operand): A[row 8jt+gl][k 4tig .. 4tig+3]
    uint32_t b0[J], b1[J];
#pragma unroll
    for (int jt = 0; jt < J; ++jt) lds64(st + L::kA + (8 * jt + gl) * 32 + 8 * tig, b0[jt], b1[jt]);

    // packed weights: rows 4tig+r, this lane's V words
    uint32_t w[4][V];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if constexpr (V == 1) {
        w[r][0] = lds32(st + w_off[r]);
      } else if constexpr (V == 2) {
        lds64(st + w_off[r], w[r][0], w[r][1]);
      } else {
        lds128(st + w_off[r], w[r][0], w[r][1], w[r][2], w[r][3]);
      }
    }

#pragma unroll
    for (int v = 0; v < V; ++v) {
      // h[pair][j]: pair 0 = rows (4tig, 4tig+1), pair 1 = rows (4tig+2, 4tig+3); column 8(V gl + v) + j
      uint32_t h[2][8];
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const uint32_t lo = prmt(w[2 * pr][v], w[2 * pr + 1][v], 0x5410);  // nibbles 0..3 of both rows
        const uint32_t hi = prmt(w[2 * pr][v], w[2 * pr + 1][v], 0x7632);  // nibbles 4..7 of both rows
        if constexpr (BF) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            h[pr][j] = and_or(lo >> (4 * j), 0x000F000Fu, 0x43004300u);
            h[pr][j + 4] = and_or(hi >> (4 * j), 0x000F000Fu, 0x43004300u);
          }
        } else {
          const uint32_t lo8 = lo >> 8, hi8 = hi >> 8;
          h[pr][0] = and_or(lo, 0x000F000Fu, 0x64006400u);
          h[pr][1] = and_or(lo, 0x00F000F0u, 0x54005400u);
          h[pr][2] = and_or(lo8, 0x000F000Fu, 0x64006400u);
          h[pr][3] = and_or(lo8, 0x00F000F0u, 0x54005400u);
          h[pr][4] = and_or(hi, 0x000F000Fu, 0x64006400u);
          h[pr][5] = and_or(hi, 0x00F000F0u, 0x54005400u);
          h[pr][6] = and_or(hi8, 0x000F000Fu, 0x64006400u);
          h[pr][7] = and_or(hi8, 0x00F000F0u, 0x54005400u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) h[pr][j] = mul2_rn<BF>(sub2_rn<BF>(h[pr][j], zsub[v][j]), s2[v][j]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // MMA rows: gl -> column 8(V gl + v) + q ; gl + 8 -> column 8(V gl + v) + q + 4
        const uint32_t af[4] = {h[0][q], h[0][q + 4], h[1][q], h[1][q + 4]};
#pragma unroll
        for (int jt = 0; jt < J; ++jt) mma_16816<BF>(acc[jt][v][q], af, b0[jt], b1[jt]);
      }
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncthreads();  // every warp is done with its ring: the ring area becomes the reduction buffer

  // ---- reduction: warps (shared memory), then cluster ranks (distributed shared memory) ----
  float *red = reinterpret_cast<float *>(smem);  // [kWarps][kMT][kWN]
  constexpr int kTile = L::kMT * L::kWN;
#pragma unroll
  for (int jt = 0; jt < J; ++jt)
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int n = 8 * (V * gl + v) + q;
        const int m = 8 * jt + 2 * tig;
        float *base = red + warp * kTile;
        base[m * L::kWN + n] = acc[jt][v][q][0];
        base[(m + 1) * L::kWN + n] = acc[jt][v][q][1];
        base[m * L::kWN + n + 4] = acc[jt][v][q][2];
        base[(m + 1) * L::kWN + n + 4] = acc[jt][v][q][3];
      }
  __syncthreads();

  const int64_t rows_here = min64(L::kMT, p.M - m0);
  for (int o = threadIdx.x; o < kTile; o += blockDim.x) {
    if (o / L::kWN < rows_here) {
      float s = 0.f;
#pragma unroll
      for (int wi = 0; wi < kWarps; ++wi) s += red[wi * kTile + o];
      red[o] = s;
    }
  }

  auto store = [&](int o, float v) {
    const int m = o / L::kWN, n = o % L::kWN;
    const int64_t gn = n0 + n;
    if (m < rows_here && gn < p.N) {
      if (p.bias) v += bits_to_float(p.bias[gn], BF);
      const T y = DT::from_float_rn(v);
      p.out[(m0 + m) * p.N + gn] = *reinterpret_cast<const uint16_t *>(&y);
    }
  };

  if (C == 1) {
    __syncthreads();
    for (int o = threadIdx.x; o < kTile; o += blockDim.x) store(o, red[o]);
  } else {
    cluster_sync_all();  // every rank's CTA sum is complete and visible cluster-wide
    const int per = (kTile + C - 1) / C;
    const int o_begin = rank * per, o_end = o_begin + per < kTile ? o_begin + per : kTile;
    const uint32_t red_u32 = smem_u32(red);
    for (int o = o_begin + threadIdx.x; o < o_end; o += blockDim.x) {
      if (o / L::kWN < rows_here) {
        float s = 0.f;
        for (int rr = 0; rr < C; ++rr) s += ld_dsmem_f32(map_to_rank(red_u32 + 4u * o, rr));
        store(o, s);
      }
    }
    cluster_sync_all();  // keep this CTA's shared memory alive until every rank has read it
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
using KernelFn = void (*)(const DecodeParams);

template <class DT, int V, int J, bool Z>
KernelFn kernel_ptr() {
  return decode_kernel<DT, V, J, Z>;
}
template <int V, int J, bool Z>
int smem_bytes() {
  return DecodeLayout<V, J, Z>::kSmem;
}

struct Variant {
  KernelFn fn;
  int smem;
};

template <class DT, bool Z>
Variant pick_vj(int V, int J) {
  if (J == 1) {
    if (V == 1) return {kernel_ptr<DT, 1, 1, Z>(), smem_bytes<1, 1, Z>()};
    return {kernel_ptr<DT, 2, 1, Z>(), smem_bytes<2, 1, Z>()};
  }
  if (J == 2) return {kernel_ptr<DT, 1, 2, Z>(), smem_bytes<1, 2, Z>()};
  return {kernel_ptr<DT, 1, 4, Z>(), smem_bytes<1, 4, Z>()};
}

Variant pick(int dtype, bool has_zp, int V, int J) {
  if (dtype == W4A16_BF16) return has_zp ? pick_vj<BF16, true>(V, J) : pick_vj<BF16, false>(V, J);
  return has_zp ? pick_vj<F16, true>(V, J) : pick_vj<F16, false>(V, J);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool decode_supported(const GemmArgs &g) {
  return g.N % 32 == 0 && g.K % 16 == 0 && g.group_size % 16 == 0 && aligned16(g.a) &&
         aligned16(g.b_q) && aligned16(g.scales) && (g.qzeros == nullptr || aligned16(g.qzeros));
}

void decode_make_plan(int64_t M, int64_t K, int64_t N, int has_zp, int num_sms, w4a16_plan_t *p) {
  const int J = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
  const int64_t KS = K / 16;
  const int64_t m_tiles = (M + 8 * J - 1) / (8 * J);
  // Two CTAs of 8 warps fit on an SM (registers and shared memory): aim for one such wave.
  const int64_t slots = 2 * int64_t(num_sms);
  int bestV = 1, bestC = 1;
  double best = -1.0;
  for (int V = 2; V >= 1; --V) {
    if (J > 1 && V != 1) continue;  // multi-tile rows: one word per lane keeps registers in check
    const int64_t n_tiles = (N + 64 * V - 1) / (64 * V);
    for (int C = 1; C <= 8; ++C) {
      if (C > 1 && KS < int64_t(C) * kWarps) break;  // every warp keeps at least one k-step
      const int64_t ctas = n_tiles * C * m_tiles;
      const int64_t waves = (ctas + slots - 1) / slots;
      double eff = double(ctas) / double(waves * slots);
      if (V == 2) eff *= 1.08;  // wider loads and fewer column tiles: preferred at equal fill
      if (eff > best + 1e-9) {
        best = eff;
        bestV = V;
        bestC = C;
      }
    }
  }
  const int V = bestV;
  const int64_t C = bestC;
  const int64_t n_tiles = (N + 64 * V - 1) / (64 * V);
  const int64_t kc = (KS + C - 1) / C;
  p->path = W4A16_PATH_DECODE;
  p->words_per_lane = V;
  p->m_tile = 8 * J;
  p->n_tile = 64 * V;
  p->k_split = static_cast<int32_t>(C);
  p->warps = kWarps;
  p->grid = n_tiles * C * m_tiles;
  p->smem_bytes = pick(W4A16_F16, has_zp != 0, V, J).smem;
  p->reserved = static_cast<int32_t>(kc);
}

cudaError_t launch_gemm_decode(const GemmArgs &g, const w4a16_plan_t &pl) {
  const int V = pl.words_per_lane, J = pl.m_tile / 8, C = pl.k_split;
  const Variant var = pick(g.dtype, g.qzeros != nullptr, V, J);

  static std::mutex mu;
  static bool configured[64][2][2][5] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    const int vi = V == 1 ? (J == 1 ? 0 : (J == 2 ? 3 : 4)) : 1;
    std::lock_guard<std::mutex> lock(mu);
    bool &done = configured[dev & 63][g.dtype == W4A16_BF16][g.qzeros != nullptr][vi];
    if (!done) {
      e = cudaFuncSetAttribute(var.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, var.smem);
      if (e != cudaSuccess) return e;
      done = true;
    }
  }

  DecodeParams prm;
  prm.a = static_cast<const uint16_t *>(g.a);
  prm.b_q = g.b_q;
  prm.scales = static_cast<const uint16_t *>(g.scales);
  prm.qzeros = g.qzeros;
  prm.bias = static_cast<const uint16_t *>(g.bias);
  prm.out = static_cast<uint16_t *>(g.out);
  prm.M = g.M;
  prm.K = g.K;
  prm.N = g.N;
  prm.G = g.group_size;
  prm.zp_bias = g.zp_bias;
  prm.k_split = C;
  const int64_t KS = g.K / 16;
  prm.ksteps_per_cta = static_cast<int>((KS + C - 1) / C);

  const int64_t n_tiles = (g.N + 64 * V - 1) / (64 * V);
  const int64_t m_tiles = (g.M + 8 * J - 1) / (8 * J);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_tiles * C), static_cast<unsigned>(m_tiles), 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(var.smem);
  cfg.stream = g.stream;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  if (C > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = static_cast<unsigned>(C);
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  e = cudaLaunchKernelEx(&cfg, var.fn, prm);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

}  // namespace w4a16

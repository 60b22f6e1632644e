// Prefill path of the W4A16 product (large M): a TMA-fed tcgen05 GEMM that dequantises int4 weight
// tiles into shared memory right before the tensor cores consume them.
//
// The pages' prefill kernel is a Triton tile loop (PR #51453 report, implementation breakdown: tile
// BLOCK_M/N/K chosen at run time, BLOCK_K clamped to the group size; PR #40977 report, key source
// snippets: fp32 accumulator, dequantise then multiply-add per K tile). On sm_103a this becomes:
//
//  * CTA tile 128*MT (rows of A; MT = 1 or 2 accumulators) x 256 (output columns), K in blocks of
//    64. Work is a list of (tile, K block) units, split three ways (the host plan picks by a cost
//    model): one CTA per tile; persistent stream-K, each CTA an equal contiguous share of the units,
//    partial tiles meeting through the caller's workspace; or, for 128-row problems, the C CTAs of a
//    thread-block cluster splitting one tile's K blocks, partial tiles meeting in distributed shared
//    memory. 10 warps per CTA:
//      warp 0      TMA producer: A tile (128x64, 128-byte swizzle), packed weight tile (64 rows x 32
//                  words), the one or two scale rows and zero-point rows the block needs;
//      warp 1      TMEM allocator and the single MMA-issuing thread;
//      warps 2..9  dequantisers, then the epilogue.
//  * Dequantisation: each thread owns one packed word column (8 output columns) and 8 rows of the
//    block; per word one LOP3 per output pair puts nibbles j and j+4 into the low mantissa bits of a
//    packed fp16 (exponent of 1024, or 64 for high nibbles) or bf16 (exponent of 128) pair, an exact
//    subtraction of (base + zp) yields q - zp, one packed multiply by the scale rounds once: exactly
//    the value w4a16_dequant writes. The 16-byte result (columns n, n+4, n+1, n+5, ...) goes to the
//    shared-memory B tile in the MN-major 128-byte-swizzled layout the tensor core reads; the epilogue
//    undoes the column interleave.
//  * MMA: tcgen05.mma.cta_group::1.kind::f16, M=128, N=256, K=16, one per 128-row half of the
//    tile, fp32 accumulators in 256*MT TMEM columns; A K-major, B MN-major. Each dequantised B tile
//    feeds MT MMAs, so MT = 2 halves the dequantisation work per FLOP. tcgen05.commit frees stages.
//  * Pipelines, each stage with full/empty mbarriers. MT = 2: 3 stages of A, freed by the MMAs'
//    commit, and 3 stages of packed weights with their scale and zero-point rows, freed by the
//    dequantisers as soon as the words are in registers. MT = 1: 5 stages holding both, freed by
//    both. 3 stages of dequantised B. Every wait is bounded (default 2 s, settable for tests): on
//    expiry the CTA records an error word, stops, drains its own TMA copies and MMAs with a fixed
//    bound, frees its TMEM and exits without writing output.
//  * Epilogue: tcgen05.ld 32 columns at a time (double-buffered), + bias in fp32, one rounding to
//    the dtype, 32-byte stores when aligned (PR #40977 report, key source snippets, test reference:
//    bias before the cast). Split tiles: contributors publish fp32 partials (stream-K: workspace;
//    cluster: own shared memory); the tile owner (stream-K) or every rank (cluster, a share each)
//    adds them in CTA order, so results do not depend on timing.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int BN = 256, BK = 64;
constexpr int64_t kPBytesHost = BK * (BN / 8) * 4;  // one packed 64 x 256 block
constexpr int kDequantWarps = 8;
constexpr int kThreads = 32 * (2 + kDequantWarps);

// MT accumulators of 128 rows each: the CTA tile is 128*MT rows x 256 columns, and each
// dequantised weight tile feeds MT MMAs.
template <int MT>
struct PLayout {
  static constexpr int BM = 128 * MT;
  // TMA rings. MT = 2: A (freed by the MMAs that read it) and the packed weights with their scale and
  // zero-point rows (freed by the dequantisers as soon as they hold them in registers) in separate
  // rings, so a weight block is requested without waiting for the MMAs three blocks back. MT = 1: one
  // ring of (A, weights) stages freed by both; measured faster there (by 20 % on 5120 x 7168) than
  // separate rings of any depth tried.
  static constexpr bool kShared = MT == 1;
  static constexpr int SA = MT == 1 ? 5 : 3;   // stages of A
  static constexpr int SP = kShared ? SA : 3;  // stages of packed weights / scales / zeros
  static constexpr int SB = 3;                 // stages of dequantised weights
  // MT = 1: the dequantisers work in two groups of 4 warps on alternate K blocks (a group's waits,
  // fence and arrivals overlap the other group's arithmetic); MT = 2: all 8 warps on every block.
  static constexpr int kDqGroups = MT == 1 ? 2 : 1;
  static constexpr int kGroupWarps = kDequantWarps / kDqGroups;
  static constexpr uint32_t kTmemCols = 256u * MT;
  static constexpr int kABytes = BM * BK * 2;        // 16 KB per 128 rows
  static constexpr int kPBytes = BK * (BN / 8) * 4;  // 8 KB
  static constexpr int kSBytes = 2 * BN * 2;         // up to two scale rows
  static constexpr int kZBytes = 2 * (BN / 8) * 4;   // up to two zero-point rows
  static constexpr int kBBytes = BK * BN * 2;        // 32 KB
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + SA * kABytes;
  static constexpr int kOffP = kOffB + SB * kBBytes;
  static constexpr int kOffS = kOffP + SP * kPBytes;
  static constexpr int kOffZ = kOffS + SP * kSBytes;
  static constexpr int kOffBar = kOffZ + SP * kZBytes;
  // stream-K fix-up: after the last MMA the A and B stage buffers stage contributors' partial tiles,
  // 32 KB chunks (one epilogue column chunk of all eight warps)
  static constexpr int kFixChunk = 32768;
  static constexpr int kFixSlots = (kOffP - kOffA) / kFixChunk;
  // + accumulator full/empty, epilogue done, stall test, fix-up ready, fix-up slot full/empty,
  // accumulators released (teardown)
  static constexpr int kNumBars = 2 * SA + 2 * SB + (kShared ? 0 : 2 * SP) + 6 + 2 * kFixSlots;
  static constexpr int kOffSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffFlag = kOffSlot + 4;
  static constexpr int kSmemUsed = kOffFlag + 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 bytes
  static_assert(kOffB % 1024 == 0 && kBBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
// Stream-K workspace: the per-CTA "partial ready" flags first, at a fixed place (so that no plan's
// partial tiles ever cover another plan's flags), then one fp32 partial tile per CTA.
constexpr size_t kFlagBytes = 4096;
constexpr int64_t kMaxStreamKCtas = kFlagBytes / 4;

__device__ unsigned int g_prefill_error;
__device__ unsigned long long g_wait_limit_ns;
__device__ unsigned int g_prefill_stall;  // test hook: dequantisers first wait on a barrier nobody arrives on

// ---------------------------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, tcgen05
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32-byte global store (sm_100+ vector width), 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&o)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]),
               "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
               : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 in bits 0-13, leading byte offset >> 4 in
// 16-29, stride byte offset >> 4 in 32-45, the fixed 0b001 in 46-48, swizzle mode in 61-63
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

struct PrefillParams {
  const uint16_t *bias;
  uint16_t *out;
  int64_t M, K, N;
  int G;
  int g_shift;       // log2(G) when G is a power of two; otherwise G == K and every row is in group 0 (31)
  int zp_bias;
  int nk;            // K blocks of 64
  int m_tiles;       // row tiles
  int n_tiles;       // column tiles
  int64_t tiles;     // m_tiles x n_tiles; tile t covers row tile t % m_tiles and column tile
                     // t / m_tiles, or (column tiles fastest) column tile t % n_tiles and row tile t / n_tiles
  float *partials;   // stream-K: one fp32 [BM][BN] partial tile per CTA (null when every CTA owns whole tiles)
  unsigned int *flags;  // stream-K: per-CTA "partial ready" flags; zero before and after every launch
  int csplit;        // > 1: clusters of csplit CTAs split each tile's K blocks (128-row tiles only)
  int a_rows;        // rows of A per TMA box: BM, or M rounded up to 8 when one row tile covers M
  int dp_waves;      // stream-K: whole waves of tiles done data-parallel first (CTA c: c, c + G, ...)
  const uint8_t *b_pp;    // prepacked weights (null: b_q through the tensor map)
  int64_t pp_tile_bytes;  // bytes of one column tile's blocks in the prepacked layout
};

// First (tile, K block) work unit of CTA c when the tiles x nk units are split evenly over G CTAs.
__device__ __forceinline__ int64_t unit_begin(int64_t c, int64_t total, int64_t G) { return c * total / G; }

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned int *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned int *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <bool BF>
__device__ __forceinline__ void magic4(uint32_t w, uint32_t (&h)[4]) {
  // h[i] = packed (base + nibble i, base + nibble i+4) with an exact integer in the low mantissa bits
  if constexpr (BF) {
    h[0] = and_or(w, 0x000F000Fu, 0x43004300u);
    h[1] = and_or(w >> 4, 0x000F000Fu, 0x43004300u);
    h[2] = and_or(w >> 8, 0x000F000Fu, 0x43004300u);
    h[3] = and_or(w >> 12, 0x000F000Fu, 0x43004300u);
  } else {
    const uint32_t w8 = w >> 8;
    h[0] = and_or(w, 0x000F000Fu, 0x64006400u);   // 1024 + q
    h[1] = and_or(w, 0x00F000F0u, 0x54005400u);   // 64 + q (high nibble of a byte, ulp 1/16)
    h[2] = and_or(w8, 0x000F000Fu, 0x64006400u);
    h[3] = and_or(w8, 0x00F000F0u, 0x54005400u);
  }
}

// COLS: consecutive tiles step along the column tiles instead of the row tiles (see the work split).
template <class DT, bool HAS_ZP, bool TWO_GROUPS, int MT, bool COLS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmP,
                   const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                   const PrefillParams p) {
  constexpr bool BF = DT::kBF16;
  using L = PLayout<MT>;
  constexpr int BM = L::BM, SA = L::SA, SB = L::SB, SP = L::SP;
  constexpr bool kShared = L::kShared;
  constexpr int kDqGroups = L::kDqGroups, kGroupWarps = L::kGroupWarps;
  constexpr int kABytes = L::kABytes, kPBytes = L::kPBytes, kSBytes = L::kSBytes, kZBytes = L::kZBytes,
                kBBytes = L::kBBytes;
  constexpr int kOffA = L::kOffA, kOffB = L::kOffB, kOffP = L::kOffP, kOffS = L::kOffS, kOffZ = L::kOffZ,
                kOffBar = L::kOffBar, kOffSlot = L::kOffSlot, kOffFlag = L::kOffFlag;
  constexpr uint32_t kTmemCols = L::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t *base_ptr = smem_raw + (base - raw_u32);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work units are (tile, K block) pairs. Stream-K plans first run dp_waves whole waves of tiles
  // data-parallel: CTA c takes tiles c, c + G, c + 2G, ..., so the CTAs of a wave step through K
  // together over neighbouring tiles and share the A and weight slices in L2. A wave sweeps the whole
  // faster tile dimension, so the host makes that the dimension of the smaller operand (row tiles
  // when A is the smaller, column tiles - COLS - when the weights are): the operand swept by every
  // wave then stays in L2 and the larger one is read from HBM about once.
  // The remaining tiles' units, tile-major, are then split into contiguous, even shares (with one CTA
  // per tile every share is a whole tile): a share may start or end inside a tile; the CTA holding a
  // tile's K block 0 owns it and adds the partial tiles of the CTAs that hold the rest (they publish
  // them in the workspace) before the epilogue.
  const int nk = p.nk;
  const int64_t G = gridDim.x;
  // Cluster split-K: the C CTAs of a cluster share one tile, rank r taking K blocks
  // [r nk / C, (r + 1) nk / C); their partial tiles meet in distributed shared memory.
  const int C = p.csplit;
  const int64_t dp_tiles = C > 1 ? 0 : int64_t(p.dp_waves) * G;  // tiles done data-parallel
  const int dp_units = C > 1 ? 0 : p.dp_waves * nk;              // this CTA's data-parallel units
  const int64_t total = (p.tiles - dp_tiles) * nk;                // units shared out after them
  // this CTA's share, in units counted from the first shared tile
  const int64_t u_begin = C > 1 ? (blockIdx.x / C) * int64_t(nk) + int64_t(blockIdx.x % C) * nk / C
                                : unit_begin(blockIdx.x, total, G);
  const int64_t u_end = C > 1 ? (blockIdx.x / C) * int64_t(nk) + int64_t(blockIdx.x % C + 1) * nk / C
                              : unit_begin(int64_t(blockIdx.x) + 1, total, G);
  const int n_units = dp_units + static_cast<int>(u_end - u_begin);
  const int kb_first = static_cast<int>(u_begin % nk);
  // The share's last segment needs a fix-up when it starts a tile (K block 0) but ends inside it: the
  // CTAs after this one hold the rest of that tile and publish their partial tiles.
  const int64_t s_first = u_begin / nk;  // first and last shared tile, counted from dp_tiles
  const int64_t s_last = u_end > u_begin ? (u_end - 1) / nk : s_first;
  const bool fix_needed =
      C == 1 && u_end > u_begin && (s_last > s_first || kb_first == 0) && u_end < (s_last + 1) * nk;
  int64_t c_fix = blockIdx.x;  // last CTA holding part of tile s_last
  if (fix_needed)
    while (c_fix + 1 < G && unit_begin(c_fix + 1, total, G) < (s_last + 1) * nk) ++c_fix;
  const int n_con = static_cast<int>(c_fix - blockIdx.x);  // contributors to add
  // Tile and K block of this CTA's units, walked in order by every role (no division per unit: the
  // single MMA-issuing and producer threads are on the critical path): start at unit 0, then step.
  // The cursor also carries the tile's row and column tile indices, kept up to date by additions: the
  // producer needs both every unit. The faster of the two wraps at F tiles into the slower one.
  struct Cursor {
    int64_t t;
    int kb;
    int mt;      // row tile
    int64_t nt;  // column tile
  };
  const int F = COLS ? p.n_tiles : p.m_tiles;
  auto cursor_at = [&](int64_t t, int kb) {
    if constexpr (COLS) return Cursor{t, kb, static_cast<int>(t / F), t % F};
    else return Cursor{t, kb, static_cast<int>(t % F), t / F};
  };
  const int g_fr = static_cast<int>(G % F);  // a data-parallel step of G tiles: within and across F
  const int64_t g_fq = G / F;
  const Cursor cur0 = dp_units > 0 ? cursor_at(int64_t(blockIdx.x), 0) : cursor_at(dp_tiles + s_first, kb_first);
  const Cursor cur_shared = cursor_at(dp_tiles + s_first, kb_first);
  auto step = [&](Cursor &c, int i_next) {  // from unit i_next - 1 to unit i_next
    if (i_next == dp_units) {
      c = cur_shared;  // the data-parallel tiles are done: the shared ones
    } else if (++c.kb == nk) {
      c.kb = 0;
      if constexpr (COLS) {
        if (i_next < dp_units) {
          c.t += G;
          c.nt += g_fr;
          c.mt += static_cast<int>(g_fq);
        } else {
          c.t += 1;
          c.nt += 1;
        }
        if (c.nt >= F) {
          c.nt -= F;
          c.mt += 1;
        }
      } else {
        if (i_next < dp_units) {
          c.t += G;
          c.mt += g_fr;
          c.nt += g_fq;
        } else {
          c.t += 1;
          c.mt += 1;
        }
        if (c.mt >= F) {
          c.mt -= F;
          c.nt += 1;
        }
      }
    }
  };

  const uint32_t bar0 = base + kOffBar;
  auto full_a = [&](int s) { return bar0 + 8u * s; };
  auto empty_a = [&](int s) { return bar0 + 8u * (SA + s); };
  auto full_b = [&](int s) { return bar0 + 8u * (2 * SA + s); };
  auto empty_b = [&](int s) { return bar0 + 8u * (2 * SA + SB + s); };
  // with a shared ring the weight barriers are the A barriers
  auto full_p = [&](int s) { return kShared ? full_a(s) : bar0 + 8u * (2 * SA + 2 * SB + s); };
  auto empty_p = [&](int s) { return kShared ? empty_a(s) : bar0 + 8u * (2 * SA + 2 * SB + SP + s); };
  const uint32_t accum_full = bar0 + 8u * (2 * SA + 2 * SB + (kShared ? 0 : 2 * SP));
  const uint32_t accum_empty = accum_full + 8u;
  const uint32_t epi_done = accum_empty + 8u;  // the epilogue warps' stores of a split tile are done
  const uint32_t stall_bar = epi_done + 8u;
  const uint32_t fix_ready = stall_bar + 8u;  // committed after this CTA's last MMA
  constexpr int kFixSlots = L::kFixSlots;
  auto fix_full = [&](int s) { return fix_ready + 8u * (1 + s); };
  auto fix_empty = [&](int s) { return fix_ready + 8u * (1 + kFixSlots + s); };
  const uint32_t tmem_done = fix_ready + 8u * (1 + 2 * kFixSlots);  // every epilogue warp is past TMEM
  const uint32_t abort_flag = base + kOffFlag;
  const uint32_t slot = base + kOffSlot;

  const unsigned long long lim = g_wait_limit_ns;
  const uint64_t limit_ns = lim ? lim : kDefaultWaitNs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(empty_a(s), kShared ? kGroupWarps + 1 : 1);  // shared: the dequantisers and the MMAs
    }
    if constexpr (!kShared) {
      for (int s = 0; s < SP; ++s) {
        mbar_init(full_p(s), 1);
        mbar_init(empty_p(s), kGroupWarps);
      }
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(full_b(s), kGroupWarps);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(accum_empty, kDequantWarps);
    mbar_init(epi_done, kDequantWarps);
    mbar_init(stall_bar, 1);
    mbar_init(fix_ready, 1);
    for (int s = 0; s < kFixSlots; ++s) {
      mbar_init(fix_full(s), 1);
      mbar_init(fix_empty(s), kDequantWarps);
    }
    mbar_init(tmem_done, kDequantWarps);
    st_flag(abort_flag, 0u);
    mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    // descriptors live in the kernel parameters, not in memory an earlier kernel writes
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmP);
    prefetch_tensormap(&tmS);
    if constexpr (HAS_ZP) prefetch_tensormap(&tmZ);
  }
  if (warp == 1) tmem_alloc(slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Inputs may come from the previous kernel of the stream: wait for it before the first global
  // access, then let the next kernel begin launching.
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(base_ptr + kOffSlot);

  constexpr int srows = TWO_GROUPS ? 2 : 1;  // G = 32: a K block spans two scale groups

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // With a single row tile only the rows up to M (rounded up to 8) are fetched; the MMA still reads
      // BM rows of the stage, and the stale rows past them only reach accumulator rows past M, which
      // nothing stores (row m of the product depends on row m of A alone).
      const uint32_t tx_a = uint32_t(p.a_rows) * (BK * 2);
      const uint32_t tx_p = kPBytes + srows * (BN * 2) + (HAS_ZP ? srows * (BN / 8) * 4 : 0);
      // Split rings: unit j's weights are requested kLag units before its A block. Iteration j waits
      // for the weight slot of unit j (freed by the dequantisers of unit j - SP) and the A slot of
      // unit j - kLag (freed by the MMAs of unit j - kLag - SA = j - SP), so neither wait holds up the
      // other ring in steady state, and every wait depends only on work already requested.
      constexpr int kLag = kShared ? 0 : SP - SA;
      int issued_p = 0, issued_a = 0;
      Cursor cp = cur0, ca = cur0;
      auto issue_a = [&](int j) -> bool {  // units in order: j == issued_a
        const int s = j % SA;
        if (!wait_phase(empty_a(s), ((j / SA) & 1) ^ 1u, abort_flag, limit_ns, &g_prefill_error)) return false;
        if (j > 0) step(ca, j);
        mbar_arrive_expect_tx(full_a(s), tx_a);
        tma_load_2d(base + kOffA + s * kABytes, &tmA, ca.kb * BK, ca.mt * BM, full_a(s));
        issued_a = j + 1;
        return true;
      };
      bool run = true;
      for (int j = 0; j < n_units && run; ++j) {
        const int s = j % SP;
        if (j > 0) step(cp, j);
        const int kbp = cp.kb;
        run = wait_phase(empty_p(s), ((j / SP) & 1) ^ 1u, abort_flag, limit_ns, &g_prefill_error);
        if (!run) break;
        if constexpr (kShared) {
          // one stage, one barrier: A and the weights of unit j together
          mbar_arrive_expect_tx(full_a(s), tx_a + tx_p);
          tma_load_2d(base + kOffA + s * kABytes, &tmA, kbp * BK, cp.mt * BM, full_a(s));
          issued_a = j + 1;
        } else {
          mbar_arrive_expect_tx(full_p(s), tx_p);
        }
        const int n0 = static_cast<int>(cp.nt * BN);
        const int k0 = kbp * BK;
        const int grow = k0 >> p.g_shift;
        if (p.b_pp)  // prepacked: the block is 8 KB of contiguous words (rows with permuted chunks)
          bulk_load(base + kOffP + s * kPBytes, p.b_pp + cp.nt * p.pp_tile_bytes + int64_t(kbp) * kPBytes,
                    kPBytes, full_p(s));
        else
          tma_load_2d(base + kOffP + s * kPBytes, &tmP, n0 / 8, k0, full_p(s));
        tma_load_2d(base + kOffS + s * kSBytes, &tmS, n0, grow, full_p(s));
        if constexpr (HAS_ZP) tma_load_2d(base + kOffZ + s * kZBytes, &tmZ, n0 / 8, grow, full_p(s));
        issued_p = j + 1;
        if (!kShared && j >= kLag) run = issue_a(j - kLag);
      }
      if constexpr (!kShared)
        for (int j = issued_a; j < n_units && run; ++j) run = issue_a(j);
      if (ld_flag(abort_flag)) {
        // let this CTA's own copies land before its shared memory is released
        for (int i = issued_p - 1; i >= 0 && i >= issued_p - SP; --i) drain_phase(full_p(i % SP), (i / SP) & 1, &g_prefill_error);
        if constexpr (!kShared)
          for (int i = issued_a - 1; i >= 0 && i >= issued_a - SA; --i) drain_phase(full_a(i % SA), (i / SA) & 1, &g_prefill_error);
      } else if (fix_needed) {
        // Fix-up loader: once the last MMA is done the stage buffers are free; wait for each
        // contributor's "partial ready" flag, then stream their partial tiles, chunk by chunk in
        // the order the epilogue adds them (column chunk major, CTA order within a chunk).
        bool ok = wait_phase(fix_ready, 0, abort_flag, limit_ns, &g_prefill_error);
        const uint64_t t0 = globaltimer();
        for (int64_t cc = int64_t(blockIdx.x) + 1; cc <= c_fix && ok; ++cc) {
          while (ld_acquire_u32(p.flags + cc) == 0u) {
            if (ld_flag(abort_flag) || globaltimer() - t0 > limit_ns) {
              st_flag(abort_flag, 1u);
              atomicOr(&g_prefill_error, 1u);
              ok = false;
              break;
            }
          }
        }
        fence_proxy_async_all();  // the partials were written by other CTAs' generic stores
        const int n_chunks = 4 * MT * n_con;
        int fix_issued = 0;
        for (int n = 0; n < n_chunks && ok; ++n) {
          const int sl = n % kFixSlots;
          if (n >= kFixSlots)
            ok = wait_phase(fix_empty(sl), ((n / kFixSlots) & 1) ^ 1u, abort_flag, limit_ns, &g_prefill_error);
          if (!ok) break;
          const int it = n / n_con;
          const int64_t cc = int64_t(blockIdx.x) + 1 + (n - it * n_con);
          const float *src = p.partials + (cc * (4 * MT) + it) * (L::kFixChunk / 4);
          mbar_arrive_expect_tx(fix_full(sl), L::kFixChunk);
          bulk_load(base + kOffA + sl * L::kFixChunk, src, L::kFixChunk, fix_full(sl));
          fix_issued = n + 1;
        }
        if (!ok) {
          for (int n = fix_issued - 1; n >= 0 && n >= fix_issued - kFixSlots; --n)
            drain_phase(fix_full(n % kFixSlots), (n / kFixSlots) & 1, &g_prefill_error);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = (1u << 4)                         // D: fp32
                             | ((BF ? 1u : 0u) << 7)           // A: f16 / bf16
                             | ((BF ? 1u : 0u) << 10)          // B: f16 / bf16
                             | (0u << 15)                      // A K-major
                             | (1u << 16)                      // B MN-major
                             | (uint32_t(BN >> 3) << 17)       // N
                             | (uint32_t(128 >> 4) << 24);     // M (one MMA per 128-row half)
      bool ok = true;
      int seg = 0;
      bool seg_start = true;
      Cursor cm = cur0;
      for (int i = 0; i < n_units && ok; ++i) {
        const int sa = i % SA, sb = i % SB;
        if (i > 0) step(cm, i);
        const int kb = cm.kb;
        if (seg_start && seg > 0) {
          // the epilogue of the previous segment has read the accumulators out of TMEM
          ok = wait_phase(accum_empty, (seg - 1) & 1, abort_flag, limit_ns, &g_prefill_error);
          if (!ok) break;
        }
        ok = wait_phase(full_a(sa), (i / SA) & 1, abort_flag, limit_ns, &g_prefill_error) &&
             wait_phase(full_b(sb), (i / SB) & 1, abort_flag, limit_ns, &g_prefill_error);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_base = base + kOffA + sa * kABytes;
        const uint32_t b_base = base + kOffB + sb * kBBytes;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // B: MN-major, 128-byte swizzle atoms of 64 columns x 8 rows; atoms along N 1024 B apart
          // (leading), 8-row K groups 4096 B apart (stride); a K step of 16 is two groups.
          const uint64_t bd = smem_desc(b_base + 8192u * kk, 1024u, 4096u);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; a K step of 16 is 32 bytes;
            // rows 128*mt.. start 16 KB further. Accumulator mt lives in TMEM columns 256*mt..
            const uint64_t ad = smem_desc(a_base + 16384u * mt + 32u * kk, 16u, 1024u);
            umma_f16(tmem + 256u * mt, ad, bd, idesc, (seg_start && kk == 0) ? 0u : 1u);
          }
        }
        umma_commit(empty_a(sa));
        umma_commit(empty_b(sb));
        seg_start = false;
        const bool seg_end = (kb == nk - 1) || (i == n_units - 1);
        if (seg_end) {
          umma_commit(accum_full);  // segment `seg` accumulated: hand it to the epilogue
          ++seg;
          seg_start = true;
        }
      }
      if (!ok) {
        umma_commit(accum_full);
        drain_phase(accum_full, seg & 1, &g_prefill_error);
      } else {
        umma_commit(fix_ready);  // every MMA of this CTA is done: its stage buffers are free
      }
    }
  } else {
    // ------------------------------------------------------------ dequantisers, then epilogues
    const int dw = warp - 2;  // 0..7
    const int c = lane;       // packed word column of the tile (8 output columns)
    const int pp_swz = p.b_pp ? 7 : 0;
    const int q = warp & 3;   // TMEM lane quarter this warp may read
    const int row = 32 * q + lane;
    const int half = dw >> 2;  // epilogue columns [128*half, 128*half + 128)
    bool ok = true;
    uint32_t zsub[2][4], spair[2][4];
    if constexpr (!HAS_ZP) {
      const uint32_t zb = static_cast<uint32_t>(p.zp_bias);
      // base + zp for nibbles j (low half of a byte) and j+1 (high half; fp16 uses base 64 there)
      const uint32_t lo = BF ? (0x4300u | zb) : (0x6400u | zb);
      const uint32_t hi = BF ? (0x4300u | zb) : (0x5400u | (zb << 4));
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        zsub[g][0] = zsub[g][2] = lo | (lo << 16);
        zsub[g][1] = zsub[g][3] = hi | (hi << 16);
      }
    }
    if (g_prefill_stall) {  // failure-detection test: a wait that can only run out
      ok = wait_phase(stall_bar, 0, abort_flag, limit_ns, &g_prefill_error);
      ok = __all_sync(0xffffffffu, ok);
    }
    int seg = 0, seg_kb0 = 0, epi_uses = 0;
    bool seg_open = false;  // a segment (one tile's run of K blocks) has started
    const int dgrp = dw / kGroupWarps, dwg = dw % kGroupWarps;  // dequantiser group, warp within it
    Cursor ce = cur0;
    for (int i = 0; i < n_units && ok; ++i) {
      if (i > 0) step(ce, i);
      const int64_t t = ce.t;
      const int kb = ce.kb;
      if (!seg_open) {
        seg_kb0 = kb;  // K block the segment starts at: 0 unless a share starts inside the tile
        seg_open = true;
      }
      if (i % kDqGroups == dgrp) {
        const int sp = i % SP, sb = i % SB;
        ok = wait_phase(full_p(sp), (i / SP) & 1, abort_flag, limit_ns, &g_prefill_error) &&
             wait_phase(empty_b(sb), ((i / SB) & 1) ^ 1u, abort_flag, limit_ns, &g_prefill_error);
        ok = __all_sync(0xffffffffu, ok);  // the warp leaves the loop together
        if (!ok) break;
        const uint32_t P = base + kOffP + sp * kPBytes;
        const uint32_t S = base + kOffS + sp * kSBytes;
        const uint32_t Z = base + kOffZ + sp * kZBytes;
        const uint32_t B = base + kOffB + sb * kBBytes;
        // every shared-memory load of the block first (independent, so their latencies overlap), then
        // the arithmetic and the stores
        constexpr int kRows = BK / kGroupWarps;  // rows dwg, dwg + kGroupWarps, ... of the block
        uint32_t sw[2][4], zw[2], wq[kRows];
#pragma unroll
        for (int gr = 0; gr < srows; ++gr) {
          lds128(S + gr * (BN * 2) + c * 16, sw[gr][0], sw[gr][1], sw[gr][2], sw[gr][3]);
          if constexpr (HAS_ZP) zw[gr] = lds32(Z + gr * (BN / 2) + c * 4);
        }
        // prepacked blocks hold row r's 16-byte chunk j at j ^ (r % 8); the tensor copy leaves them in order
#pragma unroll
        for (int ii = 0; ii < kRows; ++ii) {
          const int r = dwg + kGroupWarps * ii;
          wq[ii] = lds32(P + r * (BN / 2) + ((((c >> 2) ^ (r & pp_swz))) << 4) + (c & 3) * 4);
        }
        // the weight slot is free once every lane's loads have been performed (shared-memory accesses
        // of a warp complete in order, ahead of the arrive)
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_p(sp));
#pragma unroll
        for (int gr = 0; gr < srows; ++gr) {
          spair[gr][0] = prmt(sw[gr][0], sw[gr][2], 0x5410);  // (s0, s4)
          spair[gr][1] = prmt(sw[gr][0], sw[gr][2], 0x7632);  // (s1, s5)
          spair[gr][2] = prmt(sw[gr][1], sw[gr][3], 0x5410);  // (s2, s6)
          spair[gr][3] = prmt(sw[gr][1], sw[gr][3], 0x7632);  // (s3, s7)
          if constexpr (HAS_ZP) magic4<BF>(zw[gr], zsub[gr]);
        }
#pragma unroll
        for (int ii = 0; ii < kRows; ++ii) {
          const int r = dwg + kGroupWarps * ii;
          const int gr = (TWO_GROUPS && ii >= kRows / 2) ? 1 : 0;  // rows 32..63: second group
          uint32_t h[4];
          magic4<BF>(wq[ii], h);
          uint32_t x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            x[j] = mul2_rn<BF>(sub2_rn<BF>(h[j], zsub[gr][j]), spair[gr][j]);
          }
          // MN-major, 128-byte swizzle: 8-row K groups 4096 B apart, 64-column atoms 1024 B apart,
          // row r%8 at 128 B, 16-byte chunk (c%8) XOR (r%8).
          const uint32_t off = (r >> 3) * 4096u + (c >> 3) * 1024u + (r & 7) * 128u + ((((c & 7) ^ (r & 7))) << 4);
          sts128(B + off, x[0], x[1], x[2], x[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full_b(sb));
      }

      const bool seg_end = (kb == nk - 1) || (i == n_units - 1);
      if (seg_end) {
        // ---------------------------------------------------------- epilogue of this segment
        ok = wait_phase(accum_full, seg & 1, abort_flag, limit_ns, &g_prefill_error);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        tc_fence_after();
        const bool owner = seg_kb0 == 0;        // holds K block 0: adds the others' partials, stores
        const bool whole = owner && kb == nk - 1;
        const Cursor ct = cursor_at(t, 0);  // two divisions per tile, off the per-unit path
        const int64_t m0 = int64_t(ct.mt) * BM;
        const int64_t n0 = ct.nt * BN;
        // CTAs whose share starts inside this tile after this one hold the rest of it. A tile owned
        // without its end is always this CTA's last segment: the producer thread stages the
        // contributors' partial tiles (fix-up loader) once all MMAs are done.
        const int64_t c_last = (owner && !whole) ? c_fix : int64_t(blockIdx.x);
        // One 32-column chunk of the accumulators (it: accumulator mt = it / 4, chunk it % 4), already
        // loaded from TMEM into r.
        auto epi_chunk = [&](uint32_t (&r)[32], int it) {
          const int mt = it >> 2, ch = it & 3;  // accumulator (row half of the tile) and 32-column chunk
          const int tr = 128 * mt + row;        // row within the tile
          const int64_t m = m0 + tr;
          const bool row_ok = m < p.M;
          const int col0 = half * 128 + ch * 32;
          // partial tiles travel in accumulator order: chunk `it` of a CTA is 32 KB, float4 j of
          // thread (dw, lane) at ((dw * 8 + j) * 32 + lane) * 16 bytes (a warp's float4 j is 512
          // contiguous bytes)
          const uint32_t lane_off = uint32_t((dw * 8 * 32 + lane) * 16);
          if (C > 1) {
            // cluster split-K: stage this CTA's partial tile in its own (now idle) stage buffers
            const uint32_t dst = base + kOffA + it * L::kFixChunk + lane_off;
#pragma unroll
            for (int j = 0; j < 8; ++j) sts128(dst + 512u * j, r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            return;
          }
          if (!owner) {
            // publish this CTA's partial tile
            float4 *dst = reinterpret_cast<float4 *>(p.partials + (int64_t(blockIdx.x) * (4 * MT) + it) * (L::kFixChunk / 4)) +
                          lane_off / 16;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[32 * j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            return;
          }
          if (!whole) {
            // add the contributors' chunks in CTA order (deterministic), as the loader stages them
            for (int cci = 0; cci < n_con && ok; ++cci) {
              const int n = it * n_con + cci;
              const int sl = n % kFixSlots;
              ok = wait_phase(fix_full(sl), (n / kFixSlots) & 1, abort_flag, limit_ns, &g_prefill_error);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
              const uint32_t src = base + kOffA + sl * L::kFixChunk + lane_off;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint32_t x0, x1, x2, x3;
                lds128(src + 512u * j, x0, x1, x2, x3);
                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + __uint_as_float(x0));
                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + __uint_as_float(x1));
                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + __uint_as_float(x2));
                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + __uint_as_float(x3));
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(fix_empty(sl));
            }
            if (!ok) return;
          }
          // Two 8-column groups at a time: 16 outputs = 32 bytes per store (a whole sector of the
          // row) when the rows and the output pointer are 32-byte aligned; 16-byte stores otherwise.
          const bool wide = (p.N & 15) == 0 && (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
#pragma unroll
          for (int gp = 0; gp < 2 && row_ok; ++gp) {
            uint32_t o[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int g8 = 2 * gp + h;
              // accumulator columns hold outputs n+0, n+4, n+1, n+5, n+2, n+6, n+3, n+7
              float v[8];
              v[0] = __uint_as_float(r[8 * g8 + 0]);
              v[4] = __uint_as_float(r[8 * g8 + 1]);
              v[1] = __uint_as_float(r[8 * g8 + 2]);
              v[5] = __uint_as_float(r[8 * g8 + 3]);
              v[2] = __uint_as_float(r[8 * g8 + 4]);
              v[6] = __uint_as_float(r[8 * g8 + 5]);
              v[3] = __uint_as_float(r[8 * g8 + 6]);
              v[7] = __uint_as_float(r[8 * g8 + 7]);
              const int64_t n = n0 + col0 + 8 * g8;
              if (p.bias && n < p.N) {
                const uint4 bv = *reinterpret_cast<const uint4 *>(p.bias + n);
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  v[2 * e] += bits_to_float(static_cast<uint16_t>(bw[e] & 0xFFFFu), BF);
                  v[2 * e + 1] += bits_to_float(static_cast<uint16_t>(bw[e] >> 16), BF);
                }
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if constexpr (BF) {
                  const __nv_bfloat162 tt = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                  o[4 * h + e] = *reinterpret_cast<const uint32_t *>(&tt);
                } else {
                  const __half2 tt = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
                  o[4 * h + e] = *reinterpret_cast<const uint32_t *>(&tt);
                }
              }
            }
            const int64_t n = n0 + col0 + 16 * gp;  // first of the 16 columns
            uint16_t *dst = p.out + m * p.N + n;
            if (wide && n + 16 <= p.N) {
              st_global_v8(dst, o);
            } else {
              if (n < p.N) *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
              if (n + 8 < p.N) *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
        };
        auto tmem_chunk = [&](int it) {
          return tmem + (uint32_t(32 * q) << 16) + uint32_t(256 * (it >> 2) + half * 128 + (it & 3) * 32);
        };
        // A warp whose accumulator rows all lie past M has nothing to store; it skips its chunks
        // unless the stream-K exchange counts on it (contributor publishing, owner adding).
        const bool live = (C == 1 && !whole) || m0 + 32 * q < p.M;
        // TMEM loads double-buffered: chunk it + 1 is in flight while chunk it is processed
        uint32_t ra[32], rb[32];
        if (ok && live) {
          tmem_ld32(tmem_chunk(0), ra);
          tmem_wait_ld();
        }
#pragma unroll 1
        for (int it = 0; it < 4 * MT && ok && live; it += 2) {
          tmem_ld32(tmem_chunk(it + 1), rb);
          epi_chunk(ra, it);
          tmem_wait_ld();
          if (!ok) break;
          if (it + 2 < 4 * MT) tmem_ld32(tmem_chunk(it + 2), ra);
          epi_chunk(rb, it + 1);
          tmem_wait_ld();
        }
        // the accumulators have been read: the next segment's MMAs may overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accum_empty);
        // partial tiles: publish (contributor) or release the consumed flags (owner), once every
        // epilogue warp is done with its stores / reads (a bounded mbarrier wait, not a hard barrier)
        if (!whole && C == 1) {
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(epi_done);
          if (dw == 0 && lane == 0) {
            if (wait_phase(epi_done, epi_uses & 1, abort_flag, limit_ns, &g_prefill_error)) {
              if (!owner) {
                st_release_u32(p.flags + blockIdx.x, 1u);
              } else {
                for (int64_t cc = int64_t(blockIdx.x) + 1; cc <= c_last; ++cc) p.flags[cc] = 0u;
              }
            }
          }
          ++epi_uses;
        }
        if (!ok) break;
        ++seg;
        seg_open = false;
      }
    }
    // this warp's TMEM reads are complete (each tcgen05.ld was waited on): release the accumulators
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_done);
  }

  if (C > 1) {
    // Cluster split-K reduction. Every thread of every rank arrives (the roles above end without
    // early exits), so both cluster barriers complete. After the first, all ranks' staged partial
    // tiles are visible; rank r then adds its share of the tile's 8-column groups over all ranks in
    // rank order (deterministic) and stores them; the second keeps the staging alive until every
    // rank has read it.
    __syncwarp();
    cluster_sync_all();
    const int64_t t = blockIdx.x / C;
    const int r = static_cast<int>(blockIdx.x % C);
    const Cursor ct = cursor_at(t, 0);
    const int64_t m0 = int64_t(ct.mt) * BM, n0 = ct.nt * BN;
    // units: (row, 8-column group) pairs of the rows below M, rows fastest (a warp reads contiguous
    // staged float4s); rank r takes an even share
    const int nrows = static_cast<int>(p.M - m0 < BM ? p.M - m0 : BM);
    const int n_units_red = nrows * (BN / 8);
    const int u0 = r * n_units_red / C, u1 = (r + 1) * n_units_red / C;
    for (int u = u0 + static_cast<int>(threadIdx.x); u < u1; u += kThreads) {
      const int tr = u % nrows, cg = u / nrows;
      const int mt = tr >> 7, qv = (tr >> 5) & 3, ln = tr & 31;
      const int hv = cg >> 4, ch = (cg >> 2) & 3, g8 = cg & 3;
      // the staging warp of these rows and columns: (dw + 2) % 4 = quarter, dw / 4 = column half
      const int dwv = 4 * hv + ((qv + 2) & 3), it = 4 * mt + ch;
      const int64_t m = m0 + tr;
      const int64_t n = n0 + 8 * cg;
      if (n >= p.N) continue;
      // the group's raw accumulator order sits in float4 j = 2 g8 and 2 g8 + 1 of thread (dwv, ln)
      const uint32_t off = base + kOffA + it * L::kFixChunk + uint32_t(((dwv * 8 + 2 * g8) * 32 + ln) * 16);
      float4 xa[8], xb[8];
#pragma unroll
      for (int src = 0; src < 8; ++src) {
        if (src < C) {
          const uint32_t a = map_to_rank(off, static_cast<uint32_t>(src));
          xa[src] = ld_dsmem_v4(a);
          xb[src] = ld_dsmem_v4(a + 512u);
        }
      }
      float raw[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int src = 0; src < 8; ++src) {
        if (src < C) {
          raw[0] += xa[src].x; raw[1] += xa[src].y; raw[2] += xa[src].z; raw[3] += xa[src].w;
          raw[4] += xb[src].x; raw[5] += xb[src].y; raw[6] += xb[src].z; raw[7] += xb[src].w;
        }
      }
      // raw columns hold outputs n+0, n+4, n+1, n+5, n+2, n+6, n+3, n+7
      float v[8] = {raw[0], raw[2], raw[4], raw[6], raw[1], raw[3], raw[5], raw[7]};
      if (p.bias) {
        const uint4 bv = *reinterpret_cast<const uint4 *>(p.bias + n);
        const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] += bits_to_float(static_cast<uint16_t>(bw[e] & 0xFFFFu), BF);
          v[2 * e + 1] += bits_to_float(static_cast<uint16_t>(bw[e] >> 16), BF);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (BF) {
          const __nv_bfloat162 tt = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
          o[e] = *reinterpret_cast<const uint32_t *>(&tt);
        } else {
          const __half2 tt = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
          o[e] = *reinterpret_cast<const uint32_t *>(&tt);
        }
      }
      *reinterpret_cast<uint4 *>(p.out + m * p.N + n) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    cluster_sync_relaxed();
  }

  // Teardown. Warps 0 and 1 ran their roles on lane 0 only: reconverge them first. TMEM is freed
  // only once every epilogue warp has signalled (mbarrier) that its last tcgen05.ld is complete:
  // measured, the block barrier alone let warp 1 through while epilogue warps were still reading.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    drain_phase(tmem_done, 0, &g_prefill_error);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                          const PrefillParams);

template <class DT, int MT, bool COLS>
KernelFn pick_zg(bool zp, bool two) {
  if (zp) return two ? prefill_kernel<DT, true, true, MT, COLS> : prefill_kernel<DT, true, false, MT, COLS>;
  return two ? prefill_kernel<DT, false, true, MT, COLS> : prefill_kernel<DT, false, false, MT, COLS>;
}
template <class DT>
KernelFn pick_dt(bool zp, bool two, int MT, bool cols) {
  // one 128-row tile high (MT = 1) never needs the column-fastest order: its row tiles are few
  if (MT == 1) return pick_zg<DT, 1, false>(zp, two);
  return cols ? pick_zg<DT, 2, true>(zp, two) : pick_zg<DT, 2, false>(zp, two);
}
KernelFn pick(int dtype, bool zp, bool two, int MT, bool cols = false) {
  return dtype == W4A16_BF16 ? pick_dt<BF16>(zp, two, MT, cols) : pick_dt<F16>(zp, two, MT, cols);
}
int smem_of(int MT) { return MT == 2 ? PLayout<2>::kSmemBytes : PLayout<1>::kSmemBytes; }

}  // namespace

bool prefill_supported(const GemmArgs &g) {
  const int64_t tiles = ((g.M + 127) / 128) * ((g.N + BN - 1) / BN);
  return g.N % 32 == 0 && g.K % 8 == 0 && aligned16(g.a) && aligned16(g.b_pp ? g.b_pp : g.b_q) && aligned16(g.scales) &&
         aligned16(g.out) && (g.qzeros == nullptr || aligned16(g.qzeros)) && (g.bias == nullptr || aligned16(g.bias)) &&
         tiles <= 0x7fffffff;
}

size_t prefill_plan_workspace_bytes(const w4a16_plan_t &pl) {
  if (pl.path != W4A16_PATH_PREFILL || !pl.stream_k) return 0;
  // the flag area, then one fp32 partial tile per CTA
  return kFlagBytes + static_cast<size_t>(pl.grid) * pl.m_tile * BN * sizeof(float);
}

size_t prefill_workspace_bytes(int64_t M, int64_t K, int64_t N, int group_size, int num_sms) {
  w4a16_plan_t pl;
  prefill_make_plan(M, K, N, group_size, num_sms, /*workspace=*/true, /*query_device=*/false, &pl);
  return prefill_plan_workspace_bytes(pl);
}

// CTAs of the 128-row-tile kernel resident at once when launched in clusters of C: queried from the
// runtime (clusters live within a GPC), once per device and C; 0 when unknown.
static int64_t cluster_slots(int C) {
  static std::mutex mu;
  static int cache[64][9];
  static bool have[64][9] = {};
  int dev = 0;
  if (C < 2 || C > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev][C]) {
    const KernelFn fn = pick(W4A16_F16, false, false, 1);
    int n = 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_of(1)) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(C), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = static_cast<size_t>(smem_of(1));
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = static_cast<unsigned>(C);
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) == cudaSuccess) n = clusters * C;
    }
    cudaGetLastError();  // a failed query leaves no sticky state
    cache[dev][C] = n;
    have[dev][C] = true;
  }
  return cache[dev][C];
}

// Stream-K plans run whole waves of tiles data-parallel first. The remaining tiles' units are shared
// out evenly, which needs at least one unit per CTA (a CTA with an empty share would never publish
// the partial tile its tile's owner waits for): with fewer, one wave fewer runs data-parallel.
int prefill_dp_waves(int64_t tiles, int64_t nk, int64_t grid) {
  int64_t w = tiles / grid;
  const int64_t rem = tiles - w * grid;
  if (w > 0 && rem > 0 && rem * nk < grid) --w;
  return static_cast<int>(w);
}

void prefill_make_plan(int64_t M, int64_t K, int64_t N, int group_size, int num_sms, bool workspace,
                       bool query_device, w4a16_plan_t *p) {
  (void)group_size;
  // Cost in units of one (256-row tile, K block) step of the two-accumulator kernel. One CTA per SM.
  //  * one CTA per tile: waves x K blocks; a 128-row step costs 0.7 (dequantisation is not halved);
  //  * stream-K over G CTAs (needs the workspace): an even share of all steps per CTA, plus the
  //    owner's fix-up, ~3 steps per contributor whose partial tile it waits for and adds (measured);
  //  * 128-row tiles split along K over clusters of C <= 8 CTAs, partial tiles added through
  //    distributed shared memory (no workspace): waves x (K blocks / C steps + ~2 for the exchange),
  //    with the co-resident cluster count from the runtime (clusters fit within a GPC).
  const int64_t n_tiles = (N + BN - 1) / BN;
  const int64_t nk = (K + BK - 1) / BK;
  const int64_t sms = std::max(1, num_sms);
  double best = -1.0;
  int MT = 2;
  int64_t grid = 0;
  bool stream_k = false;
  int csplit = 1;
  for (int mt = 2; mt >= 1; --mt) {
    const int64_t tiles = ((M + 128 * mt - 1) / (128 * mt)) * n_tiles;
    const double cost = double((tiles + sms - 1) / sms) * double(nk) * (mt == 1 ? 0.7 : 1.0);
    if (best < 0 || cost < best - 1e-9) {
      best = cost;
      MT = mt;
      grid = tiles;
    }
  }
  // Stream-K over both tile heights (128-row steps cost 0.7, and a contributor's partial tile half).
  // Even when whole tiles fill every wave, the persistent CTAs measured equal or faster (they skip
  // the per-tile launch, prologue and pipeline fill), so the cost model alone decides.
  if (workspace) {
    for (int mt = 2; mt >= 1; --mt) {
      const int64_t tiles = ((M + 128 * mt - 1) / (128 * mt)) * n_tiles;
      const int64_t total = tiles * nk;
      const double step = mt == 1 ? 0.7 : 1.0, fix = 3.0;
      for (int64_t g = 1; g <= std::min<int64_t>(std::min<int64_t>(sms, kMaxStreamKCtas), total); ++g) {
        // whole waves data-parallel, then the remaining tiles' units in even shares
        const int64_t waves = prefill_dp_waves(tiles, nk, g), rem = tiles - waves * g;
        const int64_t share = waves * nk + (rem * nk + g - 1) / g;
        const int64_t parts = rem > 0 ? (g + rem - 1) / rem + 1 : 1;  // CTAs touching one shared tile, at most
        const double cost = double(share) * step + fix * double(parts - 1);
        if (cost < best - 1e-9) {
          best = cost;
          MT = mt;
          grid = g;
          stream_k = true;
        }
      }
    }
  }
  if (M <= 128 && nk >= 2) {
    const int64_t tiles = n_tiles;  // one 128-row tile per column tile
    for (int c = 2; c <= 8 && c <= nk; ++c) {
      int64_t slots = query_device ? cluster_slots(c) : 0;
      // without a device: GPCs of 19 SMs (GB300: 8 x 19), whole clusters per GPC
      if (slots <= 0) slots = std::max<int64_t>(1, sms / 19) * (19 / c) * c;
      if (slots <= 0) continue;
      const int64_t waves = (tiles * c + slots - 1) / slots;
      const double cost = double(waves) * (double((nk + c - 1) / c) * 0.7 + 2.0);
      if (cost < best - 1e-9) {
        best = cost;
        MT = 1;
        grid = tiles * c;
        stream_k = false;
        csplit = c;
      }
    }
  }
  p->path = W4A16_PATH_PREFILL;
  p->k_blocks_per_stage = 1;
  p->m_tile = 128 * MT;
  p->n_tile = BN;
  p->k_split = csplit;  // > 1: clusters of k_split CTAs per 128-row tile
  p->warps = kThreads / 32;
  p->grid = grid;
  p->smem_bytes = smem_of(MT);
  p->stream_k = stream_k ? 1 : 0;
}

bool prefill_weight_maps(const GemmArgs &g, WeightMaps *wm) {
  const int64_t NW = g.N / 8, ng = g.K / g.group_size;
  const bool two = g.group_size < BK && g.group_size != g.K;  // G = 32: two groups per K block
  const int srows = two ? 2 : 1;
  if (!tma_encode_2d(&wm->tS, 2, g.scales, g.N, ng, g.N * 2, BN, srows, false)) return false;
  if (g.b_pp) {
    wm->tP = wm->tS;  // unused: prepacked weights travel by plain bulk copies
  } else if (!tma_encode_2d(&wm->tP, 4, g.b_q, NW, g.K, NW * 4, BN / 8, BK, false)) {
    return false;
  }
  if (g.qzeros) {
    if (!tma_encode_2d(&wm->tZ, 4, g.qzeros, NW, ng, NW * 4, BN / 8, srows, false)) return false;
  } else {
    wm->tZ = wm->tP;  // unused
  }
  wm->key = 0;
  return true;
}

cudaError_t launch_gemm_prefill(const GemmArgs &g, const w4a16_plan_t &pl, const WeightMaps *wm) {
  const int MT = pl.m_tile / 128;
  const int BM = 128 * MT;
  const bool zp = g.qzeros != nullptr;
  const bool two = g.group_size < BK && g.group_size != g.K;  // G = 32: two groups per K block
  // one row tile: fetch only the rows up to M (rounded up to 8) of each A block
  const int a_rows = g.M <= BM ? static_cast<int>((g.M + 7) / 8 * 8) : BM;
  CUtensorMap tA;
  if (!tma_encode_2d(&tA, 2, g.a, g.K, g.M, g.K * 2, BK, a_rows, true)) return cudaErrorInvalidValue;
  WeightMaps own;
  if (!wm) {
    if (!prefill_weight_maps(g, &own)) return cudaErrorInvalidValue;
    wm = &own;
  }
  const int64_t m_tiles = (g.M + BM - 1) / BM, n_tiles = (g.N + BN - 1) / BN;
  // Consecutive tiles sweep the faster tile dimension; make it the smaller operand's (A: row tiles,
  // weights: column tiles), so that the larger operand is read from HBM about once.
  const bool cols = MT == 2 && m_tiles > 1 && g.M * g.K * 2 > g.K * g.N / 2;
  const KernelFn fn = pick(g.dtype, zp, two, MT, cols);
  {
    static std::mutex mu;
    static bool configured[64][2][2][2][2][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    bool &done = configured[dev & 63][g.dtype == W4A16_BF16][zp][two][MT - 1][cols];
    if (!done) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_of(MT));
      if (e != cudaSuccess) return e;
      done = true;
    }
  }
  PrefillParams prm;
  prm.m_tiles = static_cast<int>(m_tiles);
  prm.n_tiles = static_cast<int>(n_tiles);
  prm.tiles = m_tiles * n_tiles;
  prm.partials = nullptr;
  prm.flags = nullptr;
  if (pl.stream_k) {
    // workspace: the flag area (zero between calls), then [grid][BM][BN] fp32 partial tiles
    const size_t part_bytes = static_cast<size_t>(pl.grid) * BM * BN * sizeof(float);
    if (!g.workspace || pl.grid > kMaxStreamKCtas || g.workspace_bytes < kFlagBytes + part_bytes)
      return cudaErrorInvalidValue;
    prm.flags = static_cast<unsigned int *>(g.workspace);
    prm.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(g.workspace) + kFlagBytes);
  }
  prm.bias = static_cast<const uint16_t *>(g.bias);
  prm.out = static_cast<uint16_t *>(g.out);
  prm.M = g.M;
  prm.K = g.K;
  prm.N = g.N;
  prm.G = g.group_size;
  prm.g_shift = 31;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == g.group_size) prm.g_shift = sh;
  prm.zp_bias = g.zp_bias;
  prm.nk = static_cast<int>((g.K + BK - 1) / BK);
  prm.csplit = pl.k_split > 1 ? pl.k_split : 1;
  prm.a_rows = a_rows;
  prm.dp_waves = pl.stream_k ? prefill_dp_waves(prm.tiles, prm.nk, pl.grid) : 0;
  prm.b_pp = reinterpret_cast<const uint8_t *>(g.b_pp);
  prm.pp_tile_bytes = int64_t(prm.nk) * kPBytesHost;
  if (prm.csplit > 1 && (MT != 1 || pl.stream_k || pl.grid % prm.csplit != 0 || prm.nk < prm.csplit))
    return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_of(MT);
  cfg.stream = g.stream;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  if (prm.csplit > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = static_cast<unsigned>(prm.csplit);
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, tA, wm->tP, wm->tS, wm->tZ, prm);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

// ---------------------------------------------------------------------------------------------
// Static scratch for callers that cannot allocate device memory (w4a16_gemm_noalloc): room for the
// stream-K partial tiles of up to kStaticTiles CTAs (two 128x256 fp32 accumulators each) and their
// flags. It lives in the library's device image, so every GPU that loads the library holds it until
// the process exits, and every call shares it.
// ---------------------------------------------------------------------------------------------
constexpr size_t kStaticTiles = 160;
constexpr size_t kStaticScratchBytes = kStaticTiles * 256 * BN * sizeof(float) + 4096;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

cudaError_t prefill_static_scratch(void **ptr, size_t *bytes) {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    // once per device, with that device current: the host-side name of the array is only a
    // stand-in; the device address comes from the runtime
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  *bytes = kStaticScratchBytes;
  return cudaSuccess;
}

cudaError_t prefill_take_device_error(uint32_t *err) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(zero));
  *err = v;
  return e;
}

cudaError_t prefill_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns;
  return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof(v));
}

cudaError_t prefill_set_stall(bool on) {
  const unsigned int v = on ? 1u : 0u;
  return cudaMemcpyToSymbol(g_prefill_stall, &v, sizeof(v));
}

}  // namespace w4a16

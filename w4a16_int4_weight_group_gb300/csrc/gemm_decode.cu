// Decode / skinny path of the W4A16 product (M <= 32): a split-K GEMM that streams the packed
// weights once from HBM through TMA, dequantises them in registers and multiplies on the tensor cores.
//
// Where the ideas come from: the PR #40977 report (implementation breakdown item 3) describes a
// split-K skinny decode kernel with magic-number int4 -> half dequantisation and a cross-lane
// reduction; the PR #51453 report (review highlights) asks for split-K because small-M decode leaves
// the GPU idle. What this kernel does on sm_103a:
//
//  * Work split. A CTA owns 256 output columns and a contiguous range of K blocks (64 rows each);
//    the C CTAs of one thread-block cluster split K. Nine warps: one TMA producer and eight
//    consumers; consumer w owns columns [32w, 32w+32) of the tile. (A variant with two groups of
//    eight consumers on alternate stages is kept for tests and tuning.) Cluster ranks add their
//    partial tiles through distributed shared memory in a fixed order: deterministic, and no global
//    scratch memory.
//  * Streaming. Per K block one TMA box of packed weights (64 rows x 128 bytes, 128-byte swizzle),
//    the activation rows (8, 16 or 32 x 64, zero-filled past M), and the scale and zero-point rows of
//    the block's one or two groups land in an 8-block ring of shared-memory stages guarded by
//    full/empty mbarriers; at most 8 blocks (64 KB of weights per CTA) are requested and not yet
//    landed. With up to 16 rows a CTA takes under half of an SM, so a CTA of the next call (launched
//    early under programmatic dependent launch) is resident beside it and requests its first weights
//    before the dependency wait; with 17..32 rows a CTA takes a whole SM.
//  * Fragments. Viewing a packed row as 16-bit elements (4 nibbles = 4 consecutive columns each),
//    ldmatrix.trans delivers to lane (g, t) the element of rows 2t and 2t+1 for column quad g: the
//    two rows of a k pair side by side, which is what a 16-bit MMA register holds. The 128-byte
//    swizzle makes the eight row addresses of each 8x8 matrix hit distinct banks.
//  * Dequantisation split around the product. One LOP3 places the nibble of column j of both rows
//    of a k pair into the low mantissa bits of a packed fp16 pair with exponent of 1024 (64 for the
//    high nibble of a byte) or a bf16 pair with exponent of 128: exactly (base+q_k, base+q_k+1). One
//    packed subtraction of (base + zp) leaves q - zp, a small integer and so exact in 16 bits. The
//    tensor core multiplies these by the activations (blk = sum_k A (q - zp) in fp32); per K block
//    and group, in fp32: acc += s * blk. With up to 8 rows and one scale group per K block the
//    subtraction moves out of the loop: the MMAs take the magic values (base + q) as they are, one
//    more MMA against a ones operand gives the row sums rs = sum_k A, and at the end of a group
//    acc += s * (blk - (base + zp) * rs). The scale is applied in fp32, so the weights are never
//    rounded to 16 bits; with one-hot activations the result is exactly RNE(s * (q - zp)), the value
//    w4a16_dequant writes.
//  * Multiply. mma.sync m16n8k16 with 16 output columns as the MMA rows and up to 8 rows of A as the
//    MMA columns (the M <= 8 decode batch fills the n=8 side; 9..16 rows take two MMAs per step,
//    17..32 rows four).
//  * Epilogue. Bias is added in fp32 and the sum rounded once to the activation dtype (PR #40977
//    report, key source snippets, test reference).
//  * Every mbarrier wait is bounded: on expiry the CTA records an error word, its warps leave the
//    loop, the producer drains its own copies, and the CTA still takes part in the cluster barriers.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kBlocksPerRow = 8;               // 32-column blocks of a 256-column tile: consumer warps per group
constexpr int BN = 256;                        // output columns per CTA
constexpr int BK = 64;                         // rows of K per block
// K blocks the ring holds, per consumer-group count. One group: an 8-block ring keeps the CTA under
// half of the SM's shared memory, so a CTA of the next call can be resident beside it and fetch its
// weights before this call ends. Two groups: a 16-block ring, one CTA per SM.
#ifndef W4A16_DEC_RING1
#define W4A16_DEC_RING1 8
#endif
#ifndef W4A16_DEC_RING2
#define W4A16_DEC_RING2 16
#endif
// Zero-point handling on the tensor core: 0 = subtract (base + zp) from every weight pair before the
// MMA; 1 = multiply the magic values (base + q) and remove (base + zp) * rowsum(A) per group in fp32;
// 2 = the latter only when a K block holds one scale group. Up to 8 rows of A only (the row sums of
// a 16-row batch would not fit the registers).
#ifndef W4A16_DEC_RS
#define W4A16_DEC_RS 2
#endif
#ifndef W4A16_DEC_MINB2
#define W4A16_DEC_MINB2 1
#endif
__host__ __device__ constexpr int ring_blocks(int ncg) { return ncg == 1 ? W4A16_DEC_RING1 : W4A16_DEC_RING2; }
__host__ __device__ constexpr int threads_of(int ncg) { return 32 * (kBlocksPerRow * ncg + 1); }
// K blocks whose copies a CTA keeps in flight. A stage is requested once the stage this many blocks
// earlier has landed (and its ring slot is free): measured on GB300, 8 blocks (64 KB) per SM move a
// 25 MB layer 10 % faster than requesting a 16-block ring at once, and 4-6 blocks are slower.
constexpr int kInFlightBlocks = 8;
constexpr int kMaxCluster = 16;  // split-K factor: cluster sizes above 8 are non-portable
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

__device__ unsigned int g_decode_error;
__device__ unsigned long long g_decode_wait_limit_ns;
__device__ unsigned int g_decode_stall;  // test hook: consumers first wait on a barrier nobody arrives on

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <int J, int NCG>
struct Layout {
  static constexpr int R = ring_blocks(NCG);    // ring depth in K blocks (a power of two)
  static constexpr int kP = BK * BN / 2;        // 8 KB packed weights per K block
  static constexpr int kA = 8 * J * BK * 2;     // 1 KB per 8 rows of A per K block
  static constexpr int kS = 2 * BN * 2;         // two scale rows per K block slot
  static constexpr int kZ = 2 * (BN / 8) * 4;   // two zero-point rows per K block slot
  static constexpr int kOffP = 0;
  static constexpr int kOffA = kOffP + R * kP;
  static constexpr int kOffS = kOffA + R * kA;
  static constexpr int kOffZ = kOffS + R * kS;
  // Split-K receive buffer: this CTA's slice of the tile's partial sums from every cluster rank,
  // fp32 in groups of four, written by the ranks (this one included) with st.async: C slices of
  // ceil(512 J / C) + 3 groups, at most 8J x 256 + 16 x 16 floats. Without a cluster it holds the second
  // consumer group's partial tile instead.
  static constexpr int kRecvFloats = 8 * J * BN + 16 * kMaxCluster;
  static constexpr int kOffRecv = kOffZ + R * kZ;
  static constexpr int kOffBar = kOffRecv + kRecvFloats * 4;
  // full[R], empty[R], the stall-test barrier, the receive barrier
  static constexpr int kOffFlag = kOffBar + (2 * R + 2) * 8;
  static constexpr int kUsed = kOffFlag + 16;
  static constexpr int kSmem = kUsed + 1024;    // slack to align the base to 1024 bytes
  static_assert((R & (R - 1)) == 0 && R >= 4, "ring depth: a power of two");
  static_assert(kOffA % 1024 == 0 && kA % 1024 == 0, "swizzled tiles need 1 KB alignment");
};

struct DecodeParams {
  const uint16_t *bias;
  uint16_t *out;
  int64_t M, K, N;
  int G;
  int zp_bias;
  int k_split;      // C: CTAs per cluster along K
  int kb_per_cta;   // K blocks per cluster rank (a multiple of sb)
  int kb_total;     // K blocks of the problem
  int srows;        // scale / zero-point rows per stage
  int g_shift;      // log2(G) when a stage spans several scale groups, else 31 (one group per stage)
  int bpg;          // K blocks per scale group (1 or 2) for G in {64, 128}; 0 when a group outlasts every stage
  const uint8_t *b_pp;    // prepacked weights (null: b_q through the tensor map)
  int64_t pp_tile_bytes;  // bytes of one column tile's blocks in the prepacked layout
};

// A 16-bit float (fp16 or bf16 bits) widened exactly to fp32.
template <bool BF>
__device__ __forceinline__ float bits_to_f32(uint32_t h) {
  if constexpr (BF) return __uint_as_float(h << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Packed (base + q) pairs of the four columns of a quad from one ldmatrix.trans register
// (low half: row k, high half: row k+1, four nibbles each). base is 1024 for fp16 columns 0 and 2
// (low nibble of a byte), 64 for fp16 columns 1 and 3 (high nibble), 128 for bf16.
template <bool BF>
__device__ __forceinline__ void magic_quad(uint32_t w, uint32_t (&h)[4]) {
  if constexpr (BF) {
    h[0] = and_or(w, 0x000F000Fu, 0x43004300u);
    h[1] = and_or(w >> 4, 0x000F000Fu, 0x43004300u);
    h[2] = and_or(w >> 8, 0x000F000Fu, 0x43004300u);
    h[3] = and_or(w >> 12, 0x000F000Fu, 0x43004300u);
  } else {
    const uint32_t w8 = w >> 8;
    h[0] = and_or(w, 0x000F000Fu, 0x64006400u);
    h[1] = and_or(w, 0x00F000F0u, 0x54005400u);
    h[2] = and_or(w8, 0x000F000Fu, 0x64006400u);
    h[3] = and_or(w8, 0x00F000F0u, 0x54005400u);
  }
}
template <bool BF>
__host__ __device__ constexpr float magic_base(int j) {
  return BF ? 128.f : ((j & 1) ? 64.f : 1024.f);
}

template <class DT, int J, bool HAS_ZP, bool TWO_GROUPS, int SBS, int NCG>
__global__ void __launch_bounds__(threads_of(NCG), NCG == 1 ? (J >= 4 ? 1 : 2) : W4A16_DEC_MINB2)
    decode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmP,
                  const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                  const DecodeParams p) {
  using L = Layout<J, NCG>;
  using T = typename DT::T;
  constexpr bool BF = DT::kBF16;
  constexpr int kConsumers = kBlocksPerRow * NCG;
  constexpr int kThreads = threads_of(NCG);
  // row-sum correction instead of per-pair subtraction (see W4A16_DEC_RS)
  constexpr bool RS = J == 1 && (W4A16_DEC_RS == 1 || (W4A16_DEC_RS == 2 && !TWO_GROUPS));
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t *base_ptr = smem_raw + (base - raw_u32);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gl = lane >> 2, tig = lane & 3;

  const int C = p.k_split;
  const int rank = static_cast<int>(blockIdx.x % C);
  const int64_t n0 = int64_t(blockIdx.x / C) * BN;
  const int kb_begin = min(p.kb_total, rank * p.kb_per_cta);
  const int nkb = min(p.kb_total, kb_begin + p.kb_per_cta) - kb_begin;
  // K blocks per stage (1 or 4) and stages in the ring, both compile-time (runtime shifts here cost
  // more than the whole per-block index arithmetic they replace)
  constexpr int sbs = SBS, SB = 1 << SBS;
  constexpr int nsts = ilog2(L::R) - SBS, nst = 1 << nsts;
  const int nss = (nkb + SB - 1) >> sbs;        // stages this CTA fills

  const uint32_t full0 = base + L::kOffBar, empty0 = full0 + 8u * L::R;
  const uint32_t stall_bar = empty0 + 8u * L::R;
  const uint32_t recv_bar = stall_bar + 8u;
  // Split-K exchange across a cluster. A CTA's partial tile travels in accumulator order, four floats
  // at a time: group g = ((w * 2 + q) * J + jt) * 32 + lane holds acc[jt][q][0..3] of consumer warp w.
  // The 512 J groups are cut into C slices of per_g; rank s adds slice s over every rank. A group is
  // live when its first row 8 jt + 2 (lane & 3) lies below M; only live groups travel.
  const int64_t rows = p.M < 8 * J ? p.M : 8 * J;
  const bool push = C > 1;  // only in a cluster launch
  constexpr int kGroups4 = 512 * J;
  const int per_g = ((kGroups4 + C - 1) / C + 3) & ~3;  // a multiple of 4 (whole tig cycles)
  const int my_lo = min(kGroups4, rank * per_g), my_hi = min(kGroups4, my_lo + per_g);
  // live groups among [0, x): lanes with tig < ceil((rows - 8 jt) / 2), in 32-lane runs per jt
  auto live_below = [&](int x) {
    const int rr = static_cast<int>(rows);
    int lj[J], per_span = 0;
#pragma unroll
    for (int jt = 0; jt < J; ++jt) {
      lj[jt] = max(0, min(4, (rr - 8 * jt + 1) / 2));
      per_span += 8 * lj[jt];
    }
    int c = (x / (32 * J)) * per_span, r = x % (32 * J);
#pragma unroll
    for (int jt = 0; jt < J; ++jt) {
      const int rj = min(r, 32);
      c += (rj / 4) * lj[jt] + min(rj % 4, lj[jt]);
      r -= rj;
    }
    return c;
  };
  const int my_live = live_below(my_hi) - live_below(my_lo);
  const uint32_t abort_flag = base + L::kOffFlag;
  const unsigned long long lim = g_decode_wait_limit_ns;
  const uint64_t limit_ns = lim ? lim : kDefaultWaitNs;

  if (threadIdx.x == 0) {
    // a stage is released by the eight consumer warps of the group that reads it (the groups take
    // alternate stages)
    const uint32_t readers = kBlocksPerRow;
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, readers);
    }
    mbar_init(stall_bar, 1);
    mbar_init(recv_bar, 1);
    st_flag(abort_flag, 0u);
    mbar_init_fence();
    // every contribution to this CTA's slice lands with st.async, counted in bytes on recv_bar
    if (push) mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(C * my_live * 16));
  }
  if (warp == kConsumers && lane == 0) {
    // descriptors live in the kernel parameters, not in memory an earlier kernel writes
    prefetch_tensormap(&tmP);
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmS);
    if constexpr (HAS_ZP) prefetch_tensormap(&tmZ);
  }
  __syncthreads();
  // the peers' receive barriers are initialised before any CTA of the cluster pushes to them (this
  // runs before the dependency wait, so it overlaps the previous kernel)
  if (C > 1) cluster_sync_all();
  // Let the next kernel of the stream begin launching (it waits for this one before touching its
  // own inputs). Everything this kernel reads except the weights may come from the previous kernel.
  griddep_launch_dependents();

  float acc[J][2][4];
#pragma unroll
  for (int jt = 0; jt < J; ++jt)
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[jt][q][e] = 0.f;

  if (warp == kConsumers) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // prepacked weights: a stage's blocks are one contiguous run of 8 KB blocks, copied as they are
      // (they are stored in the order the 128-byte-swizzled tensor copy would produce)
      const uint8_t *pp_tile = p.b_pp ? p.b_pp + int64_t(blockIdx.x / C) * p.pp_tile_bytes : nullptr;
      auto stage_tx = [&](int j) {
        const int blocks = min(SB, nkb - j * SB);
        return static_cast<uint32_t>((pp_tile ? blocks : SB) * L::kP + blocks * L::kA + p.srows * BN * 2 +
                                     (HAS_ZP ? p.srows * BN / 2 : 0));
      };
      auto load_weights = [&](int j, int s) {
        const uint32_t full = full0 + 8u * s;
        const int k0 = (kb_begin + j * SB) * BK;
        const int grow = k0 / p.G;
        if (pp_tile) {
          const int blocks = min(SB, nkb - j * SB);
          bulk_load(base + L::kOffP + s * SB * L::kP, pp_tile + int64_t(kb_begin + j * SB) * L::kP,
                    static_cast<uint32_t>(blocks * L::kP), full);
        } else {
          tma_load_2d(base + L::kOffP + s * SB * L::kP, &tmP, static_cast<int>(n0 / 8), k0, full);
        }
        tma_load_2d(base + L::kOffS + s * SB * L::kS, &tmS, static_cast<int>(n0), grow, full);
        if constexpr (HAS_ZP)
          tma_load_2d(base + L::kOffZ + s * SB * L::kZ, &tmZ, static_cast<int>(n0 / 8), grow, full);
      };
      auto load_acts = [&](int j, int s) {
        const int blocks = min(SB, nkb - j * SB);
        for (int b = 0; b < blocks; ++b)
          tma_load_2d(base + L::kOffA + (s * SB + b) * L::kA, &tmA, (kb_begin + j * SB + b) * BK, 0,
                      full0 + 8u * s);
      };
      // The packed weights, scales and zero points are model parameters that no kernel of this stream
      // writes while it runs: the first ring of them is requested before waiting for the previous
      // kernel, which overlaps their latency with its tail. The activations come after the wait.
      constexpr int fl = (kInFlightBlocks >> SBS) > 0 ? (kInFlightBlocks >> SBS) : 1;  // stages in flight
      constexpr int fl_ring = nst < fl ? nst : fl;
      const int first = nss < fl_ring ? nss : fl_ring;
      for (int j = 0; j < first; ++j) {
        mbar_arrive_expect_tx(full0 + 8u * j, stage_tx(j));
        load_weights(j, j);
      }
      griddep_wait();
      for (int j = 0; j < first; ++j) load_acts(j, j);
      int issued = first;
      for (int j = first; j < nss; ++j) {
        const int s = j & (nst - 1);
        if (j >= fl) {  // the stage fl back has landed
          const int jf = j - fl;
          if (!wait_phase(full0 + 8u * (jf & (nst - 1)), (jf >> nsts) & 1, abort_flag, limit_ns, &g_decode_error)) break;
        }
        if (!wait_phase(empty0 + 8u * s, ((j >> nsts) & 1) ^ 1u, abort_flag, limit_ns, &g_decode_error)) break;
        mbar_arrive_expect_tx(full0 + 8u * s, stage_tx(j));
        load_weights(j, s);
        load_acts(j, s);
        issued = j + 1;
      }
      if (ld_flag(abort_flag)) {
        for (int j = issued - 1; j >= 0 && j >= issued - nst; --j)
          drain_phase(full0 + 8u * (j & (nst - 1)), (j >> nsts) & 1, &g_decode_error);
      }
    } else {
      griddep_wait();
    }
  } else {
    // ------------------------------------------------------------------ consumers
    griddep_wait();  // the epilogue writes `out` and reads `bias`: the previous kernel must be done
    const int grp = warp / kBlocksPerRow;  // stages grp, grp+NCG, grp+2*NCG, ...
    const int cb = warp % kBlocksPerRow;   // 16-byte chunk (32 columns) of every 128-byte packed row
    // ldmatrix row addresses: lanes 8i..8i+7 -> matrix i, row (lane & 7)
    const int mi = lane >> 3, rj = lane & 7;
    const uint32_t p_off = uint32_t((8 * mi + rj) * 128 + ((cb ^ rj) << 4));          // row blocks 0..3
    const uint32_t a_off = uint32_t(rj * 128 + ((mi ^ rj) << 4));                      // k chunks 0..3
    const uint32_t a_off2 = uint32_t(rj * 128 + (((mi + 4) ^ rj) << 4));               // k chunks 4..7
    const uint32_t s_off = uint32_t((32 * cb + 4 * gl) * 2);
    const uint32_t z_off = uint32_t((4 * cb + (gl >> 1)) * 4);
    const int z_shift = 16 * (gl & 1);
    constexpr int kSeg = TWO_GROUPS ? 2 : 1;  // scale-group segments per K block (32 rows each for G = 32)
    const bool single_row = p.M == 1;         // only accumulator column m = 0 is live

    // Column j of this lane's quad (output column n0 + 32 cb + 4 gl + j) holds magic values base_j + q
    // (magic_quad). Subtracting form: zsym[j] = (base_j + zp, base_j + zp) in the activation dtype,
    // the same unpack applied to a word whose four nibbles are the zero point. Row-sum form:
    // nzsym[j] = -(base_j + zp) in fp32.
    uint32_t zsym[4];
    float nzsym[4];
    if constexpr (!HAS_ZP) {
      magic_quad<BF>(static_cast<uint32_t>(p.zp_bias) * 0x11111111u, zsym);
#pragma unroll
      for (int j = 0; j < 4; ++j) nzsym[j] = -(magic_base<BF>(j) + static_cast<float>(p.zp_bias));
    }
    // a 16 x 16 operand of ones: its product with a block of activations is the block's row sums
    constexpr uint32_t kOnes = BF ? 0x3F803F80u : 0x3C003C00u;
    const uint32_t ones[4] = {kOnes, kOnes, kOnes, kOnes};
    bool ok = true;
    if (g_decode_stall) {  // failure-detection test: a wait that can only run out
      ok = wait_phase(stall_bar, 0, abort_flag, limit_ns, &g_decode_error);
      ok = __all_sync(0xffffffffu, ok);
    }
    // Partial products of the current scale group (fp32): blk = sum_k A[m,k] w[k,n] over the rows of
    // the group seen so far, rs = sum_k A[m,k] (row-sum form). They are scaled into acc when the
    // group ends, or when a stage ends inside it.
    float blk[J][2][4], rs[J][4];
    bool fresh = true;  // the next MMAs start blk and rs from zero
    // Products of one segment (k16 steps t0 .. t0+kSteps-1 of a K block) on the tensor core.
    // Subtracting form: one packed subtraction per pair turns (base_j + q) into q - zp, exactly (a
    // small integer). Row-sum form: the magic values go in as they are and the product with the ones
    // operand gives the row sums for the correction.
    auto products = [&](const uint32_t (&wq)[8], const uint32_t (&af)[J][8], int seg, uint32_t zraw) {
      constexpr int kSteps = TWO_GROUPS ? 2 : 4;
      uint32_t zsub[4];
      if constexpr (!RS) {
        if constexpr (HAS_ZP) {
          magic_quad<BF>(prmt(zraw, 0u, 0x1010u), zsub);  // this quad's zero points in both halves
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) zsub[j] = zsym[j];
        }
      }
#pragma unroll
      for (int tt = 0; tt < kSteps; ++tt) {
        const int t = seg * kSteps + tt;
        uint32_t lo[4], hi[4];
        magic_quad<BF>(wq[2 * t], lo);
        magic_quad<BF>(wq[2 * t + 1], hi);
        if constexpr (!RS) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            lo[j] = sub2_rn<BF>(lo[j], zsub[j]);
            hi[j] = sub2_rn<BF>(hi[j], zsub[j]);
          }
        }
        // MMA rows: g -> column 4*gl + j, g + 8 -> column 4*gl + j + 2, for j = 0 and j = 1
        const uint32_t a0[4] = {lo[0], lo[2], hi[0], hi[2]};
        const uint32_t a1[4] = {lo[1], lo[3], hi[1], hi[3]};
#pragma unroll
        for (int jt = 0; jt < J; ++jt) {
          if (fresh && tt == 0) {
            mma_16816_z<BF>(blk[jt][0], a0, af[jt][2 * t], af[jt][2 * t + 1]);
            mma_16816_z<BF>(blk[jt][1], a1, af[jt][2 * t], af[jt][2 * t + 1]);
            if constexpr (RS) mma_16816_z<BF>(rs[jt], ones, af[jt][2 * t], af[jt][2 * t + 1]);
          } else {
            mma_16816<BF>(blk[jt][0], a0, af[jt][2 * t], af[jt][2 * t + 1]);
            mma_16816<BF>(blk[jt][1], a1, af[jt][2 * t], af[jt][2 * t + 1]);
            if constexpr (RS) mma_16816<BF>(rs[jt], ones, af[jt][2 * t], af[jt][2 * t + 1]);
          }
        }
      }
      fresh = false;
    };
    // Ends a scale group: acc += s * blk (subtracting form) or acc += s * (blk - (base + zp) * rs)
    // (row-sum form), in fp32. With one-hot activations both give exactly s * (q - zp): blk and rs
    // are exact, and so are the fused multiply-adds on these small integers. With M = 1 only the
    // accumulator elements of row 0 (the even ones) are updated.
    auto flush = [&](const uint32_t (&sraw)[2], uint32_t zraw) {
      float sc[4], nz[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t h = (j < 2 ? sraw[0] : sraw[1]) >> (16 * (j & 1));
        sc[j] = bits_to_f32<BF>(h & 0xFFFFu);
      }
      if constexpr (RS) {
        if constexpr (HAS_ZP) {
          // -(base_j + zp_j): (2^23 - base_j) - (2^23 + zp_j), the second term built from the nibble
          // as the bits of a float (exact: both are integers below 2^24)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            nz[j] = (8388608.f - magic_base<BF>(j)) - __uint_as_float(0x4B000000u | ((zraw >> (4 * j)) & 0xFu));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) nz[j] = nzsym[j];
        }
      }
      auto update = [&](int jt, int q, int e) {
        const int j = q + 2 * (e >> 1);  // accumulator element e of MMA q holds column j
        if constexpr (RS) {
          const float tv = fmaf(nz[j], rs[jt][e & 1], blk[jt][q][e]);
          acc[jt][q][e] = fmaf(sc[j], tv, acc[jt][q][e]);
        } else {
          acc[jt][q][e] = fmaf(sc[j], blk[jt][q][e], acc[jt][q][e]);
        }
      };
      if (J == 1 && single_row) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          update(0, q, 0);
          update(0, q, 2);
        }
      } else {
#pragma unroll
        for (int jt = 0; jt < J; ++jt)
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) update(jt, q, e);
      }
      fresh = true;
    };
    // The group's stages, one at a time: wait for the stage, then per K block load the fragments
    // (packed weights by ldmatrix.trans, activations by ldmatrix, the block's scale and zero-point
    // words), release the stage after the last block's loads, and multiply; a scale group ends after
    // the block whose end is a multiple of G (or the stage's last block, or each 32-row half for
    // G = 32).
    for (int js = grp; js < nss && ok; js += NCG) {
      const int s = js & (nst - 1);
      ok = wait_phase(full0 + 8u * s, (js >> nsts) & 1, abort_flag, limit_ns, &g_decode_error);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int nb = min(SB, nkb - js * SB);
      const uint32_t P0 = base + L::kOffP + s * SB * L::kP;
      const uint32_t A0 = base + L::kOffA + s * SB * L::kA;
      const uint32_t S0 = base + L::kOffS + s * SB * L::kS + s_off;
      const uint32_t Z0 = base + L::kOffZ + s * SB * L::kZ + z_off;
#pragma unroll
      for (int b = 0; b < SB; ++b) {
        if (b < nb) {
          uint32_t wq[8], af[J][8], r[4];
          const uint32_t P = P0 + b * L::kP;
          ldsm_x4_trans(P + p_off, r);
          wq[0] = r[0]; wq[1] = r[1]; wq[2] = r[2]; wq[3] = r[3];
          ldsm_x4_trans(P + p_off + 4096u, r);
          wq[4] = r[0]; wq[5] = r[1]; wq[6] = r[2]; wq[7] = r[3];
#pragma unroll
          for (int jt = 0; jt < J; ++jt) {
            const uint32_t A = A0 + b * L::kA + jt * 1024u;
            ldsm_x4(A + a_off, r);
            af[jt][0] = r[0]; af[jt][1] = r[1]; af[jt][2] = r[2]; af[jt][3] = r[3];
            ldsm_x4(A + a_off2, r);
            af[jt][4] = r[0]; af[jt][5] = r[1]; af[jt][6] = r[2]; af[jt][7] = r[3];
          }
          // scale and zero-point rows of this block's group(s) within the stage's rows
          uint32_t sraw[kSeg][2], zraw[kSeg];
          const int r0 = (b * BK) >> p.g_shift;
#pragma unroll
          for (int g = 0; g < kSeg; ++g) {
            lds64(S0 + (r0 + g) * (BN * 2), sraw[g][0], sraw[g][1]);
            zraw[g] = HAS_ZP ? (lds32(Z0 + (r0 + g) * (BN / 2)) >> z_shift) : 0u;
          }
          if (b == nb - 1) {  // every value this group needs from the stage is in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * s);
          }
#pragma unroll
          for (int g = 0; g < kSeg; ++g) {
            products(wq, af, g, zraw[g]);
            // end of a scale group: every segment for G = 32; for larger G the block whose end is
            // a multiple of G; and always the stage's last block
            const int kend = kb_begin + js * SB + b + 1;  // K blocks done after this one
            if (TWO_GROUPS || b == nb - 1 || (p.bpg > 0 && (kend & (p.bpg - 1)) == 0)) flush(sraw[g], zraw[g]);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ reduction and epilogue
  __syncwarp();  // the producer warp's lanes meet again before the cluster barrier below
  auto finish = [&](int m, int64_t n, float v) {
    if (m < rows && n < p.N) {
      if (p.bias) v += bits_to_float(p.bias[n], BF);
      const T y = DT::from_float_rn(v);
      p.out[m * p.N + n] = *reinterpret_cast<const uint16_t *>(&y);
    }
  };
  const int nl0 = 32 * (warp % kBlocksPerRow) + 4 * gl;
  if (!push) {
    if constexpr (NCG == 2) {
      // one CTA: group 1 hands its sums to group 0 through shared memory (the receive buffer is free
      // without a cluster), fixed order group 0 + group 1
      float *gred = reinterpret_cast<float *>(base_ptr + L::kOffRecv);
      if (warp >= kBlocksPerRow && warp < kConsumers) {
#pragma unroll
        for (int jt = 0; jt < J; ++jt)
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) gred[(8 * jt + 2 * tig + (e & 1)) * BN + nl0 + q + 2 * (e >> 1)] = acc[jt][q][e];
      }
      // named barrier of the consumer warps only: the producer warp must not arrive on it (an extra
      // warp would open a second phase of the barrier that nobody completes)
      if (warp < kConsumers) asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
      if (warp < kBlocksPerRow) {
#pragma unroll
        for (int jt = 0; jt < J; ++jt)
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[jt][q][e] += gred[(8 * jt + 2 * tig + (e & 1)) * BN + nl0 + q + 2 * (e >> 1)];
      }
    }
    if (warp < kBlocksPerRow) {
      const int64_t nb = n0 + nl0;
#pragma unroll
      for (int jt = 0; jt < J; ++jt)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int m = 8 * jt + 2 * tig;
          finish(m, nb + q, acc[jt][q][0]);
          finish(m + 1, nb + q, acc[jt][q][1]);
          finish(m, nb + q + 2, acc[jt][q][2]);
          finish(m + 1, nb + q + 2, acc[jt][q][3]);
        }
    }
  } else {
    // Split-K across a cluster. The two consumer groups first add up in shared memory (the weight
    // ring is free once both are past their last stage), then every warp of the first group pushes
    // its live groups of four partial sums into the receive buffer of the rank that adds them, at the
    // slot of its own rank; no cluster barrier and no remote load sits between the last product and
    // the sums. A CTA that gave up a wait pushes nothing (its peers' receive waits then run out).
    const bool aborted = ld_flag(abort_flag) != 0u;
    const int cw = warp % kBlocksPerRow;
    if constexpr (NCG == 2) {
      float4 *gred = reinterpret_cast<float4 *>(base_ptr + L::kOffP);
      if (warp < kConsumers) asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
      if (warp >= kBlocksPerRow && warp < kConsumers) {
#pragma unroll
        for (int jt = 0; jt < J; ++jt)
#pragma unroll
          for (int q = 0; q < 2; ++q)
            gred[((cw * 2 + q) * J + jt) * 32 + lane] = make_float4(acc[jt][q][0], acc[jt][q][1], acc[jt][q][2], acc[jt][q][3]);
      }
      if (warp < kConsumers) asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
      if (warp < kBlocksPerRow) {
#pragma unroll
        for (int jt = 0; jt < J; ++jt)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float4 v = gred[((cw * 2 + q) * J + jt) * 32 + lane];
            acc[jt][q][0] += v.x;
            acc[jt][q][1] += v.y;
            acc[jt][q][2] += v.z;
            acc[jt][q][3] += v.w;
          }
      }
    }
    if (warp < kBlocksPerRow && !aborted) {
      const uint32_t recv0 = base + L::kOffRecv;
#pragma unroll
      for (int jt = 0; jt < J; ++jt)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (8 * jt + 2 * tig < rows) {
            const int g = ((cw * 2 + q) * J + jt) * 32 + lane;
            const int dst = g / per_g;
            const uint32_t a = recv0 + 16u * uint32_t(rank * per_g + (g - dst * per_g));
            st_async_v4(map_to_rank(a, dst), acc[jt][q][0], acc[jt][q][1], acc[jt][q][2], acc[jt][q][3],
                        map_to_rank(recv_bar, dst));
          }
        }
    }
    cluster_arrive_relaxed();
    // this CTA's slice: wait for every rank's contribution, add them in rank order, store
    bool got = my_live == 0 || wait_phase(recv_bar, 0, abort_flag, limit_ns, &g_decode_error);
    if (got) {
      const float4 *recv = reinterpret_cast<const float4 *>(base_ptr + L::kOffRecv);
      for (int i = threadIdx.x; i < my_hi - my_lo; i += kThreads) {
        const int g = my_lo + i;
        const int ln = g % 32, rest = g / 32;
        const int jt = rest % J, q = (rest / J) % 2, w = rest / (2 * J);
        const int m0 = 8 * jt + 2 * (ln & 3);
        if (m0 >= rows) continue;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < C; ++r) {
          const float4 x = recv[r * per_g + i];
          v[0] += x.x;
          v[1] += x.y;
          v[2] += x.z;
          v[3] += x.w;
        }
        const int64_t n = n0 + 32 * w + 4 * (ln >> 2) + q;
#pragma unroll
        for (int e = 0; e < 4; ++e) finish(m0 + (e & 1), n + 2 * (e >> 1), v[e]);
      }
    }
    // no CTA leaves while a peer may still push into its receive buffer
    cluster_wait();
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                          const DecodeParams);

template <class DT, int J, int SBS, int NCG>
KernelFn pick_zg(bool zp, bool two) {
  if (zp) return two ? decode_kernel<DT, J, true, true, SBS, NCG> : decode_kernel<DT, J, true, false, SBS, NCG>;
  return two ? decode_kernel<DT, J, false, true, SBS, NCG> : decode_kernel<DT, J, false, false, SBS, NCG>;
}
template <class DT, int SBS, int NCG>
KernelFn pick_j(int J, bool zp, bool two) {
  if (J == 4) {  // 17..32 rows: one consumer group only
    if constexpr (NCG == 1) return pick_zg<DT, 4, SBS, 1>(zp, two);
    return nullptr;
  }
  return J == 1 ? pick_zg<DT, 1, SBS, NCG>(zp, two) : pick_zg<DT, 2, SBS, NCG>(zp, two);
}
template <class DT, int NCG>
KernelFn pick_sb(int J, bool zp, bool two, int sb) {
  if (sb == 4) return pick_j<DT, 2, NCG>(J, zp, two);
  return sb == 2 ? pick_j<DT, 1, NCG>(J, zp, two) : pick_j<DT, 0, NCG>(J, zp, two);
}
template <class DT>
KernelFn pick_dt(int J, bool zp, bool two, int sb, int ncg) {
  return ncg == 1 ? pick_sb<DT, 1>(J, zp, two, sb) : pick_sb<DT, 2>(J, zp, two, sb);
}
KernelFn pick(int dtype, int J, bool zp, bool two, int sb, int ncg) {
  return dtype == W4A16_BF16 ? pick_dt<BF16>(J, zp, two, sb, ncg) : pick_dt<F16>(J, zp, two, sb, ncg);
}
int smem_of(int J, int ncg) {
  if (ncg == 1) return J == 1 ? Layout<1, 1>::kSmem : (J == 2 ? Layout<2, 1>::kSmem : Layout<4, 1>::kSmem);
  return J == 1 ? Layout<1, 2>::kSmem : Layout<2, 2>::kSmem;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool decode_supported_impl(const GemmArgs &g) {
  return g.M <= 32 && g.N % 32 == 0 && g.K % 8 == 0 && aligned16(g.a) && aligned16(g.b_pp ? g.b_pp : g.b_q) &&
         aligned16(g.scales) && (g.qzeros == nullptr || aligned16(g.qzeros));
}

// Test and tuning override of the decode plan (w4a16_debug_decode_override): consumer groups,
// split-K factor and K blocks per stage; 0 leaves the dispatcher's choice.
std::atomic<int> g_ovr_ncg{0}, g_ovr_c{0}, g_ovr_sb{0};

}  // namespace

void decode_set_override(int ncg, int c, int sb) {
  g_ovr_ncg.store(ncg, std::memory_order_relaxed);
  g_ovr_c.store(c, std::memory_order_relaxed);
  g_ovr_sb.store(sb, std::memory_order_relaxed);
}

// Pipeline shape for a cluster rank holding `kb` K blocks: blocks per stage (bigger TMA boxes move
// data faster, but a CTA with few blocks needs small stages to start early), and the rank's range
// rounded up to whole stages so that every stage starts on a multiple of 64 * sb rows.
static void rank_shape(int64_t kbt, int C, int *sb, int64_t *kb_per_cta, int force_sb = 0) {
  int64_t kb = (kbt + C - 1) / C;
  int b = kb >= 16 ? 4 : 1;
  if (force_sb) b = force_sb;
  kb = (kb + b - 1) / b * b;
  *sb = b;
  *kb_per_cta = kb;
}

void decode_make_plan(int64_t M, int64_t K, int64_t N, int group_size, int num_sms, bool query_device,
                      w4a16_plan_t *p) {
  (void)group_size;
  (void)query_device;
  const int J = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
  const int64_t n_tiles = (N + BN - 1) / BN;
  const int64_t kbt = (K + BK - 1) / BK;
  const double sms = double(num_sms > 0 ? num_sms : 1);
  // One consumer group per CTA (a CTA takes under half an SM, so a CTA of the next call can be
  // resident beside it and fetch its weights before this call ends). The cluster size C (split-K
  // factor) and the stage size sb minimise a cost fitted to per-call times measured on GB300 for the
  // workload layers (CUDA-graph chains of calls on rotating weight replicas; C = 1..16, stages of 1,
  // 2 and 4 blocks, M = 1 and 8): microseconds ~ (0.16 C + 0.47 kb waves + 0.45 kb over) x f, with kb
  // the K blocks per rank, waves the rounds of two CTAs per SM the grid needs, over the grid's excess
  // over one CTA per SM (in SMs) - ranks that share an SM with a rank of the same call slow down and
  // leave the next call no room to start early - and f = 0.88 for two-block stages on ranks of at
  // least 8 blocks, 0.97 on ranks of 4 to 7 (a stage wait per two blocks), 1 for one-block stages.
  // Every rank keeps at least two K blocks.
  //   With 17..32 rows (four row tiles) a CTA needs more registers and shared memory than half an SM:
  // one CTA per SM, about 0.6 us per K block, stages of one or two blocks alike, and cluster sizes
  // from {1, 2, 4, 6, 8} only (measured: clusters of 5 and 7 CTAs of this size ran 1.3-1.7x slower
  // than their share of blocks predicts). A wave holds as many CTAs as clusters of that size fit at
  // once on GB300 (measured with cudaOccupancyMaxActiveClusters for one CTA per SM: 152, 152, 144,
  // 138 and 120 of the 152 SMs for C = 1, 2, 4, 6, 8), scaled by the SM count.
  int ncg = 1;
  auto j4_capacity = [&](int C) -> double {
    const double frac = C <= 2 ? 1.0 : (C == 4 ? 144.0 / 152 : (C == 6 ? 138.0 / 152 : (C == 8 ? 120.0 / 152 : 0.0)));
    return std::floor(sms * frac / C) * C;
  };
  int bestC = 1, bestSB = 1;
  double best = -1.0;
  for (int Ct = 1; Ct <= kMaxCluster; ++Ct) {
    for (int sbt = 1; sbt <= 2; ++sbt) {
      int sb = 1;
      int64_t kb = kbt;
      rank_shape(kbt, Ct, &sb, &kb, sbt);
      const int C = static_cast<int>((kbt + kb - 1) / kb);  // ranks left after rounding to whole stages
      if (C != Ct) continue;                                 // the same plan as a smaller C
      if (C > 1 && kb < 2) continue;
      if (sb == 2 && kb < 4) continue;
      const double grid = double(n_tiles * C);
      double cost;
      if (J == 4) {
        const double cap = j4_capacity(C);
        if (cap <= 0.0) continue;
        cost = 0.16 * C + 0.6 * double(kb) * std::ceil(grid / cap);
      } else {
        const double waves = std::ceil(grid / (2.0 * sms));
        const double over = std::max(0.0, grid - sms) / sms;
        const double f = sb == 2 ? (kb >= 8 ? 0.88 : 0.97) : 1.0;
        cost = (0.16 * C + 0.47 * double(kb) * waves + 0.45 * double(kb) * over) * f;
      }
      if (best < 0 || cost < best - 1e-9) {
        best = cost;
        bestC = C;
        bestSB = sb;
      }
    }
  }
  if (const int o = g_ovr_ncg.load(std::memory_order_relaxed)) ncg = J == 4 ? 1 : o;
  if (const int oc = g_ovr_c.load(std::memory_order_relaxed)) {
    int64_t kb = kbt;
    rank_shape(kbt, oc, &bestSB, &kb, g_ovr_sb.load(std::memory_order_relaxed));
    bestC = static_cast<int>((kbt + kb - 1) / kb);
  }
  p->path = W4A16_PATH_DECODE;
  p->k_blocks_per_stage = bestSB;
  p->m_tile = 8 * J;
  p->n_tile = BN;
  p->k_split = static_cast<int32_t>(bestC);
  p->warps = kBlocksPerRow * ncg + 1;
  p->grid = n_tiles * bestC;
  p->smem_bytes = smem_of(J, ncg);
  p->stream_k = 0;
}

bool decode_supported(const GemmArgs &g) { return decode_supported_impl(g); }

bool decode_weight_maps(const GemmArgs &g, const w4a16_plan_t &pl, WeightMaps *wm) {
  const int sb = pl.k_blocks_per_stage;
  const int srows = g.group_size < BK * sb ? BK * sb / g.group_size : 1;
  const int64_t NW = g.N / 8, ng = g.K / g.group_size;
  if (!tma_encode_2d(&wm->tS, 2, g.scales, g.N, ng, g.N * 2, BN, srows, false)) return false;
  if (g.b_pp) {
    wm->tP = wm->tS;  // unused: prepacked weights travel by plain bulk copies
  } else if (!tma_encode_2d(&wm->tP, 4, g.b_q, NW, g.K, NW * 4, BN / 8, BK * sb, true)) {
    return false;
  }
  if (g.qzeros) {
    if (!tma_encode_2d(&wm->tZ, 4, g.qzeros, NW, ng, NW * 4, BN / 8, srows, false)) return false;
  } else {
    wm->tZ = wm->tP;  // unused
  }
  wm->key = sb;
  return true;
}

cudaError_t launch_gemm_decode(const GemmArgs &g, const w4a16_plan_t &pl, const WeightMaps *wm) {
  const int J = pl.m_tile / 8;
  const int C = pl.k_split;
  const int ncg = (pl.warps - 1) / kBlocksPerRow;
  const bool zp = g.qzeros != nullptr;
  const bool two = g.group_size < BK && g.group_size != g.K;  // G = 32: two groups per K block
  const int64_t kbt = (g.K + BK - 1) / BK;
  const int sb = pl.k_blocks_per_stage;
  if (sb != 1 && sb != 2 && sb != 4) return cudaErrorInvalidValue;
  // the rank's range of K blocks, rounded up to whole stages
  const int64_t kb_per_cta = ((kbt + C - 1) / C + sb - 1) / sb * sb;
  if ((kbt + kb_per_cta - 1) / kb_per_cta != C || (ncg != 1 && ncg != 2)) return cudaErrorInvalidValue;
  // scale / zero-point rows per stage: the groups of 64 * sb rows (G in {32, 64, 128} divides that
  // when it is smaller; a larger G, or G = K, leaves one group per stage)
  const int srows = g.group_size < BK * sb ? BK * sb / g.group_size : 1;
  CUtensorMap tA;
  if (!tma_encode_2d(&tA, 2, g.a, g.K, g.M, g.K * 2, BK, 8 * J, true)) return cudaErrorInvalidValue;
  WeightMaps own;
  if (!wm || wm->key != sb) {
    if (!decode_weight_maps(g, pl, &own)) return cudaErrorInvalidValue;
    wm = &own;
  }
  const KernelFn fn = pick(g.dtype, J, zp, two, sb, ncg);
  if (!fn) return cudaErrorInvalidValue;  // 17..32 rows run with one consumer group only
  const int smem = smem_of(J, ncg);
  {
    static std::mutex mu;
    static bool configured[64][2][4][2][2][3][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    bool &done = configured[dev & 63][g.dtype == W4A16_BF16][J - 1][zp][two][sb == 4 ? 2 : sb - 1][ncg - 1];
    if (!done) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      done = true;
    }
  }
  DecodeParams prm;
  prm.bias = static_cast<const uint16_t *>(g.bias);
  prm.out = static_cast<uint16_t *>(g.out);
  prm.M = g.M;
  prm.K = g.K;
  prm.N = g.N;
  prm.G = g.group_size;
  prm.zp_bias = g.zp_bias;
  prm.k_split = C;
  prm.kb_total = static_cast<int>(kbt);
  prm.kb_per_cta = static_cast<int>(kb_per_cta);
  prm.srows = srows;
  // a stage of 64 * sb rows spans several groups only for G in {32, 64, 128} below that size
  prm.g_shift = g.group_size < BK * sb ? (g.group_size == 32 ? 5 : (g.group_size == 64 ? 6 : 7)) : 31;
  // scale groups of 64 or 128 rows end on K-block boundaries; a larger group (G = K) is cut only by
  // the stage ends
  prm.bpg = (g.group_size == 64 || g.group_size == 128) ? g.group_size / BK : 0;
  prm.b_pp = reinterpret_cast<const uint8_t *>(g.b_pp);
  prm.pp_tile_bytes = kbt * int64_t(BK * BN / 2);

  const int64_t n_tiles = (g.N + BN - 1) / BN;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_tiles * C), 1, 1);
  cfg.blockDim = dim3(threads_of(ncg), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, tA, wm->tP, wm->tS, wm->tZ, prm);
  if (e != cudaSuccess) return e;
  note_launch();
  return cudaSuccess;
}

cudaError_t decode_take_device_error(uint32_t *err) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero));
  *err = v;
  return e;
}

cudaError_t decode_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns;
  return cudaMemcpyToSymbol(g_decode_wait_limit_ns, &v, sizeof(v));
}

cudaError_t decode_set_stall(bool on) {
  const unsigned int v = on ? 1u : 0u;
  return cudaMemcpyToSymbol(g_decode_stall, &v, sizeof(v));
}

}  // namespace w4a16

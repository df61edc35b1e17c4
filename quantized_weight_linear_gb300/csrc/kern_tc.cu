// Prefill (M > 16) forward on the 5th-generation tensor cores: Y = X . W_hat^T with the
// weights dequantized on the fly into tcgen05 shared-memory operands.
//
// GPTQ page ("İddia ve Gerçeklik: GPTQ") and SmoothQuant page ("Ticari Etki"): when the
// batch grows the layer becomes compute-bound and the dequantization overhead is what
// erodes weight-only speedups; W8A8 keeps both operands on the tensor cores.  Design:
//
// * CTA tile: 128 output rows x 256 tokens (each dequantized weight tile serves 256 tokens,
//   halving the dequantization per FLOP); K in blocks of 64.  W4 / W8A8: one MMA per k-step
//   with the weight tile as A (M = 128) and the X tile as B (N = 256), so D has the weight
//   rows in its TMEM lanes; SpQR in single CTAs: two MMAs per k-step (X halves as A, M = 128;
//   the weight tile as B, N = 128), tokens in the lanes (each orientation measured faster for
//   its formats);
// * SpQR with an even number of token tiles: clusters of two CTAs on consecutive token tiles of
//   one weight tile; each converts its own 64-row group and bulk-copies the converted rows
//   into the partner's stage over DSMEM (the tile is converted once per pair), with the weight
//   rows in the TMEM lanes as for W4;
// * grouped raster: consecutive CTAs take 4 token tiles of one weight tile before the next,
//   so the CTAs of a wave share weight tiles through L2;
// * warp 0: X producer -- X tiles through a 2-D tensor map (128B swizzle) into the operand
//   ring; the last warp: loader -- the packed weight units of the tile (the device image the
//   decode kernels stream; SpQR: plus the unit's outlier buckets) through cp.async.bulk into a
//   packed ring, apart from the X producer so that neither waits on the other's ring;
// * warp 1: allocates TMEM and issues tcgen05.mma (kind::f16, bf16 or fp16 operands, fp32
//   accumulators in TMEM) from one elected thread, committing each k-block back to its
//   shared-memory stage;
// * converter warps (8 for W4 and W8A8; 16 for SpQR, in two groups on alternate k-blocks in a
//   single CTA, in four groups on every fourth k-block in a pair): turn packed codes into
//   the bf16 / fp16 weight operand; for W4 / SpQR they then run the epilogue
//   (tcgen05.ld -> bf16 -> Y).  W4 and W8A8 write the operand straight into TMEM
//   (tcgen05.st, one 32-column stage of 128 lanes x 64 k per k-block, beside the accumulator)
//   and the MMA reads A from TMEM: shared memory then carries only the X tiles and the packed
//   units.  Writing the tile to shared memory and reading it back in the MMA made
//   shared-memory bandwidth the limit (measured: the same loop without conversion runs at the
//   cuBLAS rate).  SpQR builds a K-major 128B-swizzled tile in shared memory;
// * W8A8 only, 8 more warps: exactness drain -- int8 x int8 products are exact in the fp16
//   MMA, and a K chunk is cut wherever its sum could reach 2^24 (from per-block bounds: the
//   act-quant kernel's maxima of sum qx^2 and the weight tile's of sum qw^2), so the fp32
//   accumulators (TMEM columns 0..255) hold exact integers; after each chunk but the last
//   these warps split every accumulator v into v = 2^16 hi + lo (0 <= lo < 2^16), add hi into
//   a 16-bit high part kept in TMEM (columns 256..383, two tokens per column), write lo back
//   as the accumulator the next chunk continues from, and release it; after the last chunk
//   the int32 result is 2^16 high + accumulator, written as y = bf16((acc * sx) * sw) (or
//   acc).  The 16-bit high part covers every int32 result; columns 384..511 hold the weight
//   operand stages.
// Every mbarrier wait is bounded; a timeout is recorded in the workspace status word.
#include "kern_common.cuh"

namespace qlin {
namespace {

constexpr int kBN = 128, kBK = 64;
constexpr int kTileBytes = 128 * kBK * 2;  // 16 KB, one 128-row operand tile
// W8A8 exact chunks: a chunk of k-blocks is accumulated in fp32 as long as the sum of its
// blocks' bounds stays <= kExactSum.  A block's bound is ceil(sqrt(X2 W2)), X2 the largest sum
// of squared activation codes over the block among the tile's tokens and W2 the same over its
// weight rows: by Cauchy-Schwarz no token-row product sum of the block exceeds it.  A chunk
// starts from a carried low part in [0, 2^16) (see the drain), so every partial sum is an
// integer of magnitude < 2^16 + kExactSum <= 2^24 and fp32 holds it exactly.  A block's bound
// is at most 64 * 127^2, so a chunk holds at least kChunkMin = 16 blocks (1024 K).
constexpr int kExactSum = (1 << 24) - (1 << 16);
constexpr int kChunkMin = 16;
static_assert(kChunkMin * 64 * 127 * 127 <= kExactSum, "kChunkMin blocks always fit one chunk");

// an upper bound of ceil(sqrt(x2 w2)): both < 2^24 are exact in fp32, the product and the
// square root each round by at most 2^-24 relative, the 2^-20 margin covers both
__device__ __forceinline__ int block_bound(int32_t x2, uint32_t w2) {
  return (int)(sqrtf((float)x2 * (float)w2) * 1.00000095f) + 1;
}

constexpr int kOutCapTc = 1024;            // SpQR outlier entries staged per (unit, row group)
constexpr int kOffsCapTc = 1040;           // SpQR bucket offsets staged per row group
#ifndef QLIN_TC_RASTER_G
#define QLIN_TC_RASTER_G 4
#endif
constexpr int kRasterG = QLIN_TC_RASTER_G;  // token tiles per raster group

enum Fmt { kW4 = 0, kSpqr = 1, kW8 = 2 };

// Ring depths (compile-time knobs; defaults measured on GB300 at M = 4096, K = 8192,
// N = 28672): X/B operand stages and packed-unit stages per format.
#ifndef QLIN_W8_NPK
#define QLIN_W8_NPK 4
#endif
#ifndef QLIN_W4_ATMEM
#define QLIN_W4_ATMEM 1
#endif
#ifndef QLIN_W4_ST
#define QLIN_W4_ST 4
#endif
#ifndef QLIN_W8_ATMEM
#define QLIN_W8_ATMEM 1
#endif
#ifndef QLIN_W8_ST
#define QLIN_W8_ST (QLIN_W8_ATMEM ? 4 : 3)
#endif
#ifndef QLIN_W8_CONV
#define QLIN_W8_CONV 8
#endif
#ifndef QLIN_W4_NPK
#define QLIN_W4_NPK 3
#endif
#ifndef QLIN_SP_NPK
#define QLIN_SP_NPK 2
#endif
#ifndef QLIN_SP_GROUPS
#define QLIN_SP_GROUPS 2
#endif
#ifndef QLIN_W8_PLAN_PAR
#define QLIN_W8_PLAN_PAR 1
#endif
#ifndef QLIN_SP_PAIR_ST
#define QLIN_SP_PAIR_ST 4
#endif
#ifndef QLIN_TC_SPQR_PAIRS
#define QLIN_TC_SPQR_PAIRS 1
#endif
#ifndef QLIN_W4_CONV
#define QLIN_W4_CONV 8
#endif
#ifndef QLIN_W4_GROUPS
#define QLIN_W4_GROUPS 1
#endif

template <int F>
struct TcCfg;
template <>
struct TcCfg<kW4> {
  static constexpr int kUnitBytes = kW4UnitBytes, kBlocksPerUnit = 2, kMH = 2, kConv = QLIN_W4_CONV, kStages = QLIN_W4_ST;
  static constexpr int kConvGroups = QLIN_W4_GROUPS;
  static constexpr int kNPK = QLIN_W4_NPK;  // packed-unit stages (each covers kBlocksPerUnit k-blocks)
  static constexpr uint32_t kAType = 1;  // bf16
  static constexpr bool kRowsInLanes = true;  // D = weight rows (TMEM lanes) x tokens (columns)
  static constexpr bool kATmem = QLIN_W4_ATMEM;  // converted weights go to TMEM, not shared memory
};
template <>
struct TcCfg<kSpqr> {
  static constexpr int kUnitBytes = kSpqrUnitBytes, kBlocksPerUnit = 4, kMH = 2, kConv = 16, kStages = 3;
  static constexpr int kConvGroups = QLIN_SP_GROUPS;  // two groups of 8 converter warps take alternate k-blocks
  static constexpr int kNPK = QLIN_SP_NPK;
  static constexpr uint32_t kAType = 1;
  static constexpr bool kRowsInLanes = false;  // D = tokens (lanes) x weight rows (columns); pairs: see the kernel
  static constexpr bool kATmem = false;
};
template <>
struct TcCfg<kW8> {
  static constexpr int kUnitBytes = kW8UnitBytes, kBlocksPerUnit = 1, kMH = 2, kConv = QLIN_W8_CONV, kStages = QLIN_W8_ST;
  static constexpr int kConvGroups = 1;
  static constexpr int kNPK = QLIN_W8_NPK;  // a W8 unit covers one k-block: prefetch deeper
  static constexpr uint32_t kAType = 0;  // fp16
  static constexpr bool kRowsInLanes = true;  // (the drain epilogue assumes this)
  static constexpr bool kATmem = QLIN_W8_ATMEM;
};

// CL: a CTA of a pair stages the packed units, outliers and offsets of its one row group, and
// spends the room on one more operand stage
template <int F, bool CL = false>
struct TcSmem {
  using C = TcCfg<F>;
  static constexpr int kStages = CL && F == kSpqr ? QLIN_SP_PAIR_ST : C::kStages;
  static constexpr int kRG = CL ? 1 : 2;  // row groups staged
  __align__(1024) uint8_t a[kStages][C::kMH * kTileBytes];
  __align__(1024) uint8_t b[kStages][C::kATmem ? 16 : kTileBytes];
  __align__(16) uint8_t pk[C::kNPK][kRG * C::kUnitBytes];
  __align__(16) uint32_t out[F == kSpqr ? C::kNPK : 1][kRG][F == kSpqr ? kOutCapTc + 8 : 4];
  __align__(16) uint32_t offs[kRG][F == kSpqr ? kOffsCapTc : 4];
  // stage releases: one barrier per k-block modulo max(stages, converter groups), see the kernel
  uint64_t ab_full[kStages], ab_empty[kStages > 4 ? kStages : 4];
  uint64_t pk_full[C::kNPK], pk_empty[C::kNPK];
  uint64_t offs_bar;
  uint64_t acc_full;
  uint64_t ch_full[2], ch_empty[2];
  uint64_t plan_full;  // W8A8: the drain warps have decided whether the tile is one exact chunk
  unsigned long long plan_sum;  // W8A8: the sum of the tile's block bounds
  int plan_one;
  uint32_t tmem;
};

struct TcArgs {
  const uint8_t* units;   // device image units
  const uint32_t* offs;   // SpQR bucket offsets
  const uint32_t* ents;   // SpQR outlier entries
  const float* sw;        // W8: per-row scales
  const float* sx;        // W8: per-token scales
  const int32_t* kbound;  // W8: [M tiles of 256][K / 64] per-block max of sum qx^2
  const uint32_t* w2;     // W8: [N tiles of 128][K / 64] per-block max of sum qw^2
  uint16_t* Y;
  int32_t* acc_out;
  int32_t* status;
  int M, N, K, RG, KU;
};

// ---- tcgen05 helpers -------------------------------------------------------------------

__device__ __forceinline__ uint64_t umma_desc_sw128(const void* smem_tile) {
  const uint64_t addr = smem_u32(smem_tile);
  uint64_t d = 0;
  d |= (addr & 0x3FFFFull) >> 4;         // start address
  d |= 1ull << 16;                       // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;      // stride byte offset: 8 rows x 128 B
  d |= 1ull << 46;                       // descriptor version (sm_100 family)
  d |= 2ull << 61;                       // 128-byte swizzle
  return d;
}

__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_type, int n, int m) {
  return (1u << 4) | (ab_type << 7) | (ab_type << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

// same, with the A operand (M rows in TMEM lanes, K packed two 16-bit values per column) read
// from tensor memory instead of shared memory
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---- a CTA pair (cluster of two) sharing one weight tile -------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the address of a shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// copy `bytes` (a multiple of 16) of this CTA's shared memory to `dst` in a CTA of the
// cluster; the copy completes as transaction bytes on the barrier at `bar` in that CTA (both
// shared::cluster addresses)
__device__ __forceinline__ void bulk_s2s_cluster(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "r"(smem_u32(src)), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// a bounded wait that acquires at cluster scope: for barriers the partner CTA arrives on
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_wait_scope(uint64_t* bar, uint32_t parity, int32_t* status) {
  if constexpr (!CLUSTER) {
    return mbar_wait(bar, parity, status);
  } else {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
      if (mbar_try_wait_cluster(bar, parity)) return true;
      if (global_ns() - t0 > kWaitLimitNs) break;
    }
    if (status) atomicExch(status, kStatusTimeout);
    return false;
  }
}

// commit to the same barrier in both CTAs of the pair
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// byte offset of element (row, k) in a 128 x 64 K-major tile with 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int row, int k) {
  return (uint32_t)(row * 128 + ((((k >> 3) ^ row) & 7) << 4) + ((k & 7) << 1));
}

__device__ __forceinline__ void sts32(uint8_t* base, uint32_t off, uint32_t v) {
  *reinterpret_cast<uint32_t*>(base + off) = v;
}

// Swizzled byte offsets of one converter lane's stores, computed once.  A converter writes
// 16-row tiles whose first row is a multiple of 16, so for its rows g and g + 8 the row's
// low three bits are g and sw128() reduces to XOR-ing the 16-byte chunk index with g: every
// store address is then a per-lane base plus a compile-time constant.
struct LaneSwz {
  uint32_t c[8];  // W4 / W8: (row g, k = 8c + 2t) of a tile starting at row 0
  uint32_t s[2];  // SpQR: (row g, k = 16t + 8h) for h = 0, 1
};

__device__ __forceinline__ LaneSwz lane_swz(int lane) {
  const uint32_t g = (uint32_t)lane >> 2, t = (uint32_t)lane & 3u;
  LaneSwz L;
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c) L.c[c] = g * 128u + (((c ^ g) & 7u) << 4) + 4u * t;
#pragma unroll
  for (uint32_t h = 0; h < 2; ++h) L.s[h] = g * 128u + ((((2u * t + h) ^ g) & 7u) << 4);
  return L;
}

// SpQR A-pair extraction (same field map as the decode kernel)
template <int J, int R>
__device__ __forceinline__ uint32_t sp_pair(const uint32_t (&w)[6]) {
  if constexpr (J <= 4) {
    constexpr int i = 4 * J + R;
    if constexpr (i < 18) {
      constexpr int wi = i / 3, f = (i % 3) * 2;
      return ((w[wi] >> (3 * f)) & 0x00070007u) | 0x43004300u;
    } else {
      constexpr int b = 3 * (i - 18);
      return ((w[b] >> 15) & 0x00010001u) | ((w[b + 1] >> 14) & 0x00020002u) | ((w[b + 2] >> 13) & 0x00040004u) |
             0x43004300u;
    }
  } else {
    constexpr int i = 4 * (J - 5) + R;
    constexpr int wi = i / 2, f = (i % 2) * 2 + 1;
    return ((w[wi] >> (3 * (f - 1))) & 0x00380038u) | 0x41804180u;
  }
}

__device__ __forceinline__ uint32_t sp_qsqz(const uint8_t* area, int r, int gb) {
  const int lane = 4 * (r & 7) + (gb >> 1);
  const int i = ((r >> 3) << 1) | (gb & 1);
  const int bit = 24 * lane + 6 * i;
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(area);
  return __funnelshift_r(wp[bit >> 5], wp[(bit >> 5) + 1], bit & 31) & 63u;
}

template <int J, int R0>
__device__ __forceinline__ void sp_write_j(uint8_t* bt, const uint32_t (&w)[6], uint32_t offA,
                                           uint32_t shA, uint32_t chA, uint32_t shB, uint32_t chB) {
  constexpr uint32_t base = J <= 4 ? 0x43004300u : 0x41804180u;
  // (row g, k = 16 t + 2 J) at offA + 4 (J & 3); row g + 8 is 1024 bytes further
  const uint32_t vA = bf16x2_fma(bf16x2_sub(sp_pair<J, R0>(w), base), shA, chA);
  const uint32_t vB = bf16x2_fma(bf16x2_sub(sp_pair<J, R0 + 1>(w), base), shB, chB);
  sts32(bt, offA + 4u * (J & 3), vA);
  sts32(bt, offA + 1024u + 4u * (J & 3), vB);
}

// ---- converters: one 16-row tile of the 128-row B tile for k-block kb of the packed stage

template <int F>
__device__ __forceinline__ void convert_tile(uint8_t* bt, const uint8_t* unit, int kb, int rt, int row0, int lane,
                                             bool valid, const LaneSwz& L) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t rb = (uint32_t)row0 * 128u;  // row0 is a multiple of 16
  if (!valid) {  // rows past N: zero operand
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) sts32(bt, rb + 1024u * r + L.c[kk], 0u);
    return;
  }
  if constexpr (F == kW4) {
    const uint4 wv = *reinterpret_cast<const uint4*>(unit + ((rt * 2 + kb) * 32 + lane) * 16);
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint32_t* st = reinterpret_cast<const uint32_t*>(unit + kW4CodeBytes);
    const uint32_t sz0 = st[rt * 16 + g], sz1 = st[rt * 16 + g + 8];
    const float s0 = h2f_dev((uint16_t)(sz0 & 0xFFFFu)), s1 = h2f_dev((uint16_t)(sz1 & 0xFFFFu));
    const float z0 = h2f_dev((uint16_t)(sz0 >> 16)), z1 = h2f_dev((uint16_t)(sz1 >> 16));
    const uint32_t zp0 = pack_bf16x2(128.f + z0, 128.f + z0), zp1 = pack_bf16x2(128.f + z1, 128.f + z1);
    const uint32_t sp0 = pack_bf16x2(s0, s0), sp1 = pack_bf16x2(s1, s1);
    const uint32_t zero = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // k = 16 j + 2 t (chunk 2 j) and k + 8 (chunk 2 j + 1)
      const uint32_t w = words[j];
      const uint32_t o0 = rb + L.c[2 * j], o1 = rb + L.c[2 * j + 1];
      sts32(bt, o0, bf16x2_fma(bf16x2_sub((w & 0x000F000Fu) | 0x43004300u, zp0), sp0, zero));
      sts32(bt, o0 + 1024u, bf16x2_fma(bf16x2_sub(((w >> 4) & 0x000F000Fu) | 0x43004300u, zp1), sp1, zero));
      sts32(bt, o1, bf16x2_fma(bf16x2_sub(((w >> 8) & 0x000F000Fu) | 0x43004300u, zp0), sp0, zero));
      sts32(bt, o1 + 1024u, bf16x2_fma(bf16x2_sub(((w >> 12) & 0x000F000Fu) | 0x43004300u, zp1), sp1, zero));
    }
  } else if constexpr (F == kW8) {
    const uint4 w01 = *reinterpret_cast<const uint4*>(unit + ((rt * 2 + 0) * 32 + lane) * 16);
    const uint4 w23 = *reinterpret_cast<const uint4*>(unit + ((rt * 2 + 1) * 32 + lane) * 16);
    const uint32_t words[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
    const uint32_t magic = 0x64646464u, off = 0x64806480u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // k = 16 j + 2 t (chunk 2 j) and k + 8 (chunk 2 j + 1)
      const uint32_t o0 = rb + L.c[2 * j], o1 = rb + L.c[2 * j + 1];
      uint32_t d;
      asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(d) : "r"(words[2 * j]), "r"(magic));
      sts32(bt, o0, f16x2_sub(d, off));
      asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(d) : "r"(words[2 * j]), "r"(magic));
      sts32(bt, o0 + 1024u, f16x2_sub(d, off));
      asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(d) : "r"(words[2 * j + 1]), "r"(magic));
      sts32(bt, o1, f16x2_sub(d, off));
      asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(d) : "r"(words[2 * j + 1]), "r"(magic));
      sts32(bt, o1 + 1024u, f16x2_sub(d, off));
    }
  } else {  // SpQR: k-block kb of the 256-wide unit = block kb/2, groups 4*(kb%2) .. +3
    const int blk = kb >> 1, half = kb & 1;
    const uint32_t* cw6 = reinterpret_cast<const uint32_t*>(unit) + ((rt * 2 + blk) * 32 + lane) * 6;
    uint32_t w[6];
    {
      const uint2 p0 = *reinterpret_cast<const uint2*>(cw6);
      const uint2 p1 = *reinterpret_cast<const uint2*>(cw6 + 2);
      const uint2 p2 = *reinterpret_cast<const uint2*>(cw6 + 4);
      w[0] = p0.x; w[1] = p0.y; w[2] = p1.x; w[3] = p1.y; w[4] = p2.x; w[5] = p2.y;
    }
    const uint8_t* qarea = unit + kSpqrCodeBytes + (rt * 2 + blk) * 96;
    const uint16_t* sgst = reinterpret_cast<const uint16_t*>(unit + kSpqrCodeBytes + kSpqrQsqzBytes);
    uint32_t sh[2], ch[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = g + 8 * r, gb = t + 4 * half;
      const uint16_t* st = sgst + (rt * 16 + row) * 4;
      const uint32_t e = sp_qsqz(qarea, row, gb);
      const float s_hat = __fmul_rn(__fsub_rn((float)(e & 7u), h2f_dev(st[1])), h2f_dev(st[0]));
      const float z_hat = __fmul_rn(__fsub_rn((float)(e >> 3), h2f_dev(st[3])), h2f_dev(st[2]));
      sh[r] = pack_bf16x2(s_hat, s_hat);
      const float c = -s_hat * z_hat;
      ch[r] = pack_bf16x2(c, c);
    }
    const uint32_t s0 = rb + L.s[0], s1 = rb + L.s[1];  // k = 16 t + 2 J: J < 4 -> s0, else s1
    if (half == 0) {
      sp_write_j<0, 0>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<1, 0>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<2, 0>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<3, 0>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<4, 0>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<5, 0>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<6, 0>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<7, 0>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
    } else {
      sp_write_j<0, 2>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<1, 2>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<2, 2>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<3, 2>(bt, w, s0, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<4, 2>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<5, 2>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<6, 2>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
      sp_write_j<7, 2>(bt, w, s1, sh[0], ch[0], sh[1], ch[1]);
    }
  }
}

// SpQR outliers of one (unit, row tile) bucket that fall into k-block kb, added onto the
// dequantized bf16 operand (D + s rounded once more to bf16).  Entries come from the staged
// copy when the unit's buckets fit, else from global memory.  Only the warp that wrote
// those rows touches them, and every outlier position is unique, so the read-modify-write
// is race free.
__device__ __forceinline__ void spqr_outliers_tile(uint8_t* bt, const uint32_t* staged, uint32_t stage_base,
                                                   const uint32_t* ents, uint32_t b0, uint32_t b1, int kb, int row0,
                                                   int lane) {
  // one loop per source behind a uniform branch (a select would issue the global load too)
  auto walk = [&](auto ld) {
    for (uint32_t p = b0 + lane; p < b1; p += 32) {
      const uint32_t e = ld(p);
      const int kin = (int)((e >> 4) & 255u);
      if ((kin >> 6) != kb) continue;
      const int row = row0 + (int)(e & 15u);
      uint16_t* dst = reinterpret_cast<uint16_t*>(bt + sw128(row, kin & 63));
      *dst = f2bf(__fadd_rn(bf2f(*dst), h2f_dev((uint16_t)(e >> 16))));
    }
  };
  if (staged)
    walk([&](uint32_t p) { return staged[p - stage_base]; });
  else
    walk([&](uint32_t p) { return __ldg(ents + p); });
}

template <int F>
constexpr int tc_loader_warp() {  // after the X producer, the MMA issuer, converters (+ W8A8 drains)
  return 2 + TcCfg<F>::kConv + (F == kW8 ? 8 : 0);
}

template <int F>
constexpr int tc_threads() {  // ... and the packed-unit loader
  return 32 * (tc_loader_warp<F>() + 1);
}

// 16 lanes x 32 columns from the mma.sync-style fragment: register 2r + h holds lane g + 8h,
// column 4r + t of the lane quadrant's 16-lane slice at taddr (g = lane / 4, t = lane % 4)
__device__ __forceinline__ void tmem_st16x128b_x8(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// W4 / W8 converter into TMEM: one 16-row tile, k-block kb of the packed stage, as the A
// operand of the MMA (row = TMEM lane, column c = k pair 2c, 2c + 1).  The packed fragment of
// lane (g, t) carries, per 16-wide k step j, the pairs (row g, k = 16 j + 2 t), (row g + 8,
// same k), (row g, k + 8), (row g + 8, k + 8): k pair 8 j + t and 8 j + 4 + t, i.e. columns
// 4 (2 j) + t and 4 (2 j + 1) + t, registers 4 j .. 4 j + 3 of the 16x128b.x8 store.
template <int F>
__device__ __forceinline__ void convert_tmem(uint32_t taddr, const uint8_t* unit, int kb, int rt, int lane,
                                             bool valid) {
  uint32_t v[16];
  if (!valid) {  // rows past N: zero operand
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0u;
  } else if constexpr (F == kW8) {  // offset-binary int8 codes -> fp16 (1024 + c) - 1152
    const uint4 w01 = *reinterpret_cast<const uint4*>(unit + ((rt * 2 + 0) * 32 + lane) * 16);
    const uint4 w23 = *reinterpret_cast<const uint4*>(unit + ((rt * 2 + 1) * 32 + lane) * 16);
    const uint32_t words[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
    const uint32_t magic = 0x64646464u, off = 0x64806480u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t d;
      asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(d) : "r"(words[2 * j]), "r"(magic));
      v[4 * j + 0] = f16x2_sub(d, off);
      asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(d) : "r"(words[2 * j]), "r"(magic));
      v[4 * j + 1] = f16x2_sub(d, off);
      asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(d) : "r"(words[2 * j + 1]), "r"(magic));
      v[4 * j + 2] = f16x2_sub(d, off);
      asm("prmt.b32 %0, %1, %2, 0x5342;" : "=r"(d) : "r"(words[2 * j + 1]), "r"(magic));
      v[4 * j + 3] = f16x2_sub(d, off);
    }
  } else {
    const int g = lane >> 2;
    const uint4 wv = *reinterpret_cast<const uint4*>(unit + ((rt * 2 + kb) * 32 + lane) * 16);
    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint32_t* st = reinterpret_cast<const uint32_t*>(unit + kW4CodeBytes);
    const uint32_t sz0 = st[rt * 16 + g], sz1 = st[rt * 16 + g + 8];
    const float s0 = h2f_dev((uint16_t)(sz0 & 0xFFFFu)), s1 = h2f_dev((uint16_t)(sz1 & 0xFFFFu));
    const float z0 = h2f_dev((uint16_t)(sz0 >> 16)), z1 = h2f_dev((uint16_t)(sz1 >> 16));
    const uint32_t zp0 = pack_bf16x2(128.f + z0, 128.f + z0), zp1 = pack_bf16x2(128.f + z1, 128.f + z1);
    const uint32_t sp0 = pack_bf16x2(s0, s0), sp1 = pack_bf16x2(s1, s1);
    const uint32_t zero = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w = words[j];
      v[4 * j + 0] = bf16x2_fma(bf16x2_sub((w & 0x000F000Fu) | 0x43004300u, zp0), sp0, zero);
      v[4 * j + 1] = bf16x2_fma(bf16x2_sub(((w >> 4) & 0x000F000Fu) | 0x43004300u, zp1), sp1, zero);
      v[4 * j + 2] = bf16x2_fma(bf16x2_sub(((w >> 8) & 0x000F000Fu) | 0x43004300u, zp0), sp0, zero);
      v[4 * j + 3] = bf16x2_fma(bf16x2_sub(((w >> 12) & 0x000F000Fu) | 0x43004300u, zp1), sp1, zero);
    }
  }
  tmem_st16x128b_x8(taddr, v);
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// CL (SpQR, an even number of token tiles): the two CTAs of a cluster take consecutive token
// tiles of one weight tile; each loads and converts one of its two 64-row groups and bulk-copies
// the converted rows into the partner's operand tile, so a weight tile is converted once per pair.
template <int F, bool CL = false>
__global__ void __launch_bounds__(tc_threads<F>(), 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap xmap, TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using SM = TcSmem<F, CL>;
  SM& sm = *reinterpret_cast<SM*>(base);
  using C = TcCfg<F>;
  constexpr int MH = C::kMH, NCONV = C::kConv, NST = SM::kStages;
  static_assert(!CL || F == kSpqr, "CTA pairs are built for SpQR");
  // converter warps per k-block: a pair's CTA converts 64 rows, with four groups of four warps
  // taking every fourth k-block
  constexpr int NGRP = CL ? 4 : C::kConvGroups, GCONV = NCONV / NGRP;
  // Stage releases.  The MMA commit of k-block j arrives on ab_empty[j % NEB]; whoever fills
  // k-block i's stage first waits for the commit of k-block i - NST there.  A parity wait only
  // tells a phase from the next one, so the phase before (k-block i - NST - NEB) must already be
  // known complete: the X producer and each converter group waited for exactly that commit on
  // the same barrier before their previous k-block (i - 1, resp. i - NGRP) whenever NEB is a
  // multiple of NGRP, which NEB = max(NST, NGRP) makes true for NGRP > NST.  With one barrier
  // per stage and four groups over three stages, a group two stages ahead passed the wait
  // and overwrote a stage the tensor cores had not read yet.
  constexpr int NEB = NGRP > NST ? NGRP : NST;
  static_assert(NEB <= (NST > 4 ? NST : 4), "ab_empty holds max(stages, 4) barriers");
  constexpr int BM = 128 * MH;
  constexpr int kLoaderWarp = tc_loader_warp<F>();
  const uint32_t crank = CL ? cluster_rank() : 0u, partner = crank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grouped raster: consecutive CTAs walk kRasterG token tiles of one weight tile before the
  // next weight tile, so a wave reads each weight tile from HBM once and shares it through L2
  const int mt_count = (a.M + BM - 1) / BM, nt_count = (a.N + kBN - 1) / kBN;
  const int group = (int)(blockIdx.x / (unsigned)(kRasterG * nt_count));
  const int m_first = group * kRasterG;
  const int gm = mt_count - m_first < kRasterG ? mt_count - m_first : kRasterG;
  const int r_in = (int)blockIdx.x - group * kRasterG * nt_count;
  const int m_tile = m_first + r_in % gm, n_tile = r_in / gm;
  const int64_t rg0 = (int64_t)n_tile * 2;  // two 64-row groups per 128-row tile
  const int nkb = a.K / kBK;
  const int bpu = C::kBlocksPerUnit;
  const int nunits = nkb / bpu;
  // W8A8: this tile's per-block maxima of sum qx^2 (token tile) and sum qw^2 (weight tile)
  const int32_t* kb = F == kW8 ? a.kbound + (int64_t)m_tile * nkb : nullptr;
  const uint32_t* kw = F == kW8 ? a.w2 + (int64_t)n_tile * nkb : nullptr;
  // W4, W8A8: one MMA per k-step, A = the converted weight tile (M = 128 rows), B = the X tile
  // (N = 256 tokens); D in TMEM has the weight rows in its lanes and the tokens in its columns.
  // SpQR: two MMAs per k-step, A = one 128-token half of X, B = the weight tile (N = 128); D
  // has the tokens in its lanes (measured faster for SpQR only).
  // CL: weight rows in the lanes too.  With the conversion shared by the pair, shared-memory
  // reads limit the loop, and one M = 128 x N = 256 MMA per k-step reads the weight tile once
  // where two 128-token MMAs read it twice (1.65 -> 1.48 ms at K = 8192, N = 28672; single
  // CTAs, bound by their converters, are 2% faster with the tokens in the lanes)
  constexpr bool kRowsInLanes = C::kRowsInLanes || CL;
  static_assert(F != kW8 || kRowsInLanes, "the W8A8 drain reads weight rows from TMEM lanes");
  constexpr uint32_t idesc = kRowsInLanes ? idesc_f16(C::kAType, BM, kBN) : idesc_f16(C::kAType, kBN, 128);
  // W8A8: fp32 chunk sums + int32 partials; W4: the accumulator, then one 32-column A operand
  // (128 rows x 64 k) per stage
  constexpr uint32_t tmem_cols = (F == kW8 || C::kATmem) ? 512u : 128u * MH;
  constexpr uint32_t kACol = F == kW8 ? 384u : 128u * MH;
  static_assert(!C::kATmem || (kRowsInLanes && kACol + 32u * NST <= 512u && NCONV / NGRP == 8),
                "TMEM operand stages must fit beside the accumulator; 8 converter warps per k-block");
  // SpQR: staged bucket offsets of the two row groups, global indices [4 rg S, 4 rg S + 4 S]
  int64_t off_base[2] = {0, 0};
  uint32_t off_len[2] = {0, 0};
  if constexpr (F == kSpqr) {
    for (int r = 0; r < 2; ++r) {
      const int64_t b = ((rg0 + r) * a.KU * 4) & ~int64_t(3);
      const int64_t e = ((rg0 + r) * a.KU * 4 + 4 * a.KU + 1 + 3) & ~int64_t(3);
      off_base[r] = b;
      off_len[r] = (rg0 + r < a.RG && (!CL || r == (int)crank)) ? (uint32_t)(e - b) : 0u;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&sm.ab_full[s], 1 + GCONV);  // CL: + the partner's rows as tx bytes
    for (int e = 0; e < NEB; ++e) mbar_init(&sm.ab_empty[e], CL ? 2 : 1);                    // CL: both CTAs' MMAs
    for (int s = 0; s < C::kNPK; ++s) {
      mbar_init(&sm.pk_full[s], 1);
      mbar_init(&sm.pk_empty[s], NCONV);
    }
    mbar_init(&sm.offs_bar, 1);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.plan_full, 1);
    sm.plan_sum = 0ull;
    for (int r = 0; r < 2; ++r) {
      mbar_init(&sm.ch_full[r], 1);
      mbar_init(&sm.ch_empty[r], 8);
    }
    fence_mbar_init();
    pdl_launch_dependents();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (CL) cluster_sync_all();  // the partner's barriers are initialized
  const uint32_t tmem = sm.tmem;
  bool ok = true;
  // staging slot of row group r (0 or 1 of the weight tile); a pair's CTA stages only its own
  auto slot = [&](int r) -> int { return CL ? 0 : r; };
  auto soffs = [&](int r, int64_t gi) -> uint32_t { return sm.offs[slot(r)][gi - off_base[r]]; };
  // k-block i's stage is free: the tensor cores have read k-block i - NST (both CTAs' in a pair)
  auto stage_free = [&](int i) -> bool {
    if (i < NST) return true;
    const int j = i - NST;
    return mbar_wait_scope<CL>(&sm.ab_empty[j % NEB], (uint32_t)(j / NEB) & 1u, a.status);
  };

  if (warp == kLoaderWarp) {
    // ------------------------------------------------------------------ packed-unit loader
    // Weights do not depend on the previous kernel, so this warp never waits for it.  It runs
    // apart from the X producer: the packed ring's slots are released by the converters, and
    // waiting for them in the thread that issues the X tiles would put the X load latency back
    // on every k-block.
    if (lane == 0) {
      if constexpr (F == kSpqr) {
        uint32_t bytes = 0;
        for (int r = 0; r < 2; ++r) bytes += off_len[r] * 4;
        mbar_arrive_expect_tx(&sm.offs_bar, bytes);
        for (int r = 0; r < 2; ++r)
          if (off_len[r]) bulk_g2s(sm.offs[slot(r)], a.offs + off_base[r], off_len[r] * 4, &sm.offs_bar);
        ok = mbar_wait(&sm.offs_bar, 0, a.status);
      }
      for (int ui = 0; ui < nunits && ok; ++ui) {
        const int p = ui % C::kNPK;
        const uint32_t ph = (uint32_t)(ui / C::kNPK) & 1u;
        if (!mbar_wait(&sm.pk_empty[p], ph ^ 1u, a.status)) {
          ok = false;
          break;
        }
        uint32_t bytes = 0;
        uint32_t e_lo[2] = {0, 0}, e_hi[2] = {0, 0};
        for (int r = 0; r < 2; ++r) {
          if (rg0 + r >= a.RG || (CL && r != (int)crank)) continue;
          bytes += C::kUnitBytes;
          if constexpr (F == kSpqr) {
            const int64_t u = (rg0 + r) * a.KU + ui;
            const uint32_t e0 = soffs(r, 4 * u), e1 = soffs(r, 4 * u + 4);
            if (e1 > e0 && e1 - e0 <= (uint32_t)kOutCapTc) {
              e_lo[r] = e0 & ~3u;
              e_hi[r] = (e1 + 3u) & ~3u;
              bytes += (e_hi[r] - e_lo[r]) * 4;
            }
          }
        }
        mbar_arrive_expect_tx(&sm.pk_full[p], bytes);
        for (int r = 0; r < 2; ++r) {
          if (rg0 + r >= a.RG || (CL && r != (int)crank)) continue;
          bulk_g2s(sm.pk[p] + slot(r) * C::kUnitBytes, a.units + ((rg0 + r) * a.KU + ui) * (int64_t)C::kUnitBytes,
                   C::kUnitBytes, &sm.pk_full[p]);
          if constexpr (F == kSpqr) {
            if (e_hi[r] > e_lo[r]) bulk_g2s(sm.out[p][slot(r)], a.ents + e_lo[r], (e_hi[r] - e_lo[r]) * 4, &sm.pk_full[p]);
          }
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ X producer
    pdl_wait();
    if (lane == 0) {
      for (int i = 0; i < nkb && ok; ++i) {
        const int s = i % NST;
        if (!stage_free(i)) {
          ok = false;
          break;
        }
        // CL: the partner's 64 converted rows arrive on this barrier too
        mbar_arrive_expect_tx(&sm.ab_full[s], MH * kTileBytes + (CL ? 64u * 128u : 0u));
        tma_load_2d(sm.a[s], &xmap, i * kBK, m_tile * BM, &sm.ab_full[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    pdl_wait();
    // W8A8: a tile whose bounds fit one exact chunk issues its k-blocks without any bound
    // arithmetic (the common case: chunk sizes are computed per block only otherwise).  No
    // chunk can end before k-block kChunkMin - 1, so the first blocks go out at once, and the
    // decision, which the drain warps take from the tile's block bounds meanwhile, is read
    // there.  The one-chunk path is a loop of its own with no bound bookkeeping in it: summing
    // the bounds up front delayed every tile's first MMA, and the bookkeeping inside the one
    // issue loop slowed every k-block (each cost about 8% of the kernel).
    if (lane == 0) {
      // one k-block: wait for its operands, issue its MMAs, release the stage; chunk_end
      // (W8A8) also hands the accumulators to the drain
      auto issue = [&](int i, bool chunk_end) -> bool {
        const int s = i % NST;
        if (!mbar_wait_scope<CL>(&sm.ab_full[s], (uint32_t)(i / NST) & 1u, a.status)) return false;
        tc_fence_after();
        const bool first = i == 0;
        const uint64_t dw = umma_desc_sw128(sm.b[s]);  // weights, 128 rows
        if constexpr (C::kATmem) {
          const uint64_t dx = umma_desc_sw128(sm.a[s]);  // X, 256 tokens
          const uint32_t ta = tmem + kACol + 32u * (uint32_t)s;  // weights, 128 lanes x 32 columns
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_f16_ta(tmem, ta + 8u * kk, dx + (uint64_t)(2 * kk), idesc, (first && kk == 0) ? 0u : 1u);
        } else if constexpr (kRowsInLanes) {
          const uint64_t dx = umma_desc_sw128(sm.a[s]);  // X, 256 tokens
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_f16(tmem, dw + (uint64_t)(2 * kk), dx + (uint64_t)(2 * kk), idesc, (first && kk == 0) ? 0u : 1u);
        } else {
#pragma unroll
          for (int mh = 0; mh < MH; ++mh) {
            const uint64_t dx = umma_desc_sw128(sm.a[s] + mh * kTileBytes);  // X, 128 tokens
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_f16(tmem + 128u * mh, dx + (uint64_t)(2 * kk), dw + (uint64_t)(2 * kk), idesc,
                       (first && kk == 0) ? 0u : 1u);
          }
        }
        if constexpr (CL)
          umma_commit_pair(&sm.ab_empty[i % NEB]);  // the partner's converters write this stage too
        else
          umma_commit(&sm.ab_empty[i % NEB]);
        if constexpr (F == kW8) {
          if (chunk_end) umma_commit(&sm.ch_full[0]);
        }
        return true;
      };
      int i = 0;
      if constexpr (F != kW8) {
        for (; i < nkb && ok; ++i) ok = issue(i, false);
      } else {
        const int n0 = nkb < kChunkMin - 1 ? nkb : kChunkMin - 1;
        for (; i < n0 && ok; ++i) ok = issue(i, i == nkb - 1);
        bool one_chunk = true;
        if (ok && i < nkb) {
          ok = mbar_wait(&sm.plan_full, 0u, a.status);
          one_chunk = sm.plan_one != 0;
        }
        if (one_chunk) {
          for (; i < nkb && ok; ++i) ok = issue(i, i == nkb - 1);
        } else {
          // one fp32 accumulator: chunk c starts once the drain has split chunk c - 1's
          // accumulators and written back their low parts, and continues from them.  Catch up
          // on the bounds of the blocks issued so far (i > 0 from here on).
          int bound = 0, chunk = 0;  // running bound of the current exact chunk, its index
          for (int b = 0; b < i; ++b) bound += block_bound(kb[b], kw[b]);
          int bnext = block_bound(kb[i], kw[i]);  // the next block's bound, read one k-block ahead
          for (; i < nkb && ok; ++i) {
            const int bi = bnext;
            bnext = i + 1 < nkb ? block_bound(kb[i + 1], kw[i + 1]) : 0;
            if (bound + bi > kExactSum) {
              ++chunk;
              if (!mbar_wait(&sm.ch_empty[0], (uint32_t)(chunk - 1) & 1u, a.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              bound = bi;
            } else {
              bound += bi;
            }
            ok = issue(i, i == nkb - 1 || bound + bnext > kExactSum);
          }
        }
      }
      umma_commit(&sm.acc_full);
      if constexpr (CL) {
        // commits reach both CTAs' barriers asynchronously; a converter waited for each one up to
        // k-block nkb - NST - 1 before filling the stage again.  Wait for the last NST here (the
        // partner does the same), so that no arrival is still on its way to a CTA when the pair
        // passes its final cluster barrier and leaves
        for (int i = nkb - NST > 0 ? nkb - NST : 0; i < nkb && ok; ++i)
          if (!mbar_wait_scope<CL>(&sm.ab_empty[i % NEB], (uint32_t)(i / NEB) & 1u, a.status)) ok = false;
      }
    }
    __syncwarp();
  } else if (warp < 2 + NCONV) {
    // ------------------------------------------------------------------ converters (+ epilogue)
    pdl_wait();
    const int grp = (warp - 2) / GCONV;  // this warp converts the k-blocks i with i % NGRP == grp
    const int cw = (warp - 2) % GCONV;
    constexpr int RPW = (CL ? 64 : 128) / GCONV;  // rows per converter warp: 16 or 32
    const LaneSwz swz = lane_swz(lane);
    // TMEM operand: a warp may only reach the lane quadrant warp % 4, so converter warp cw
    // takes rows 32 ((2 + cw) % 4) + 16 (cw / 4) (the group's first warp index is 2 mod 4);
    // CL: the rows of this CTA's row group
    const int row_t = C::kATmem ? 32 * ((2 + cw) % 4) + 16 * (cw / 4) : (CL ? 64 * (int)crank : 0) + cw * RPW;
    const int rg_local = row_t / 64;
    const bool rg_valid = rg0 + rg_local < a.RG;
    if constexpr (F == kSpqr) {
      if (!mbar_wait(&sm.offs_bar, 0, a.status)) ok = false;
    }
    for (int ui = 0; ui < nunits && ok; ++ui) {
      const int p = ui % C::kNPK;
      if (!mbar_wait(&sm.pk_full[p], (uint32_t)(ui / C::kNPK) & 1u, a.status)) {
        ok = false;
        break;
      }
      const uint8_t* unit = sm.pk[p] + slot(rg_local) * C::kUnitBytes;
      for (int b = 0; b < bpu; ++b) {
        const int i = ui * bpu + b;
        if (NGRP > 1 && i % NGRP != grp) continue;
        const int s = i % NST;
        if (!stage_free(i)) {
          ok = false;
          break;
        }
        if constexpr (C::kATmem) {
          tc_fence_after();
          convert_tmem<F>(tmem + ((uint32_t)row_t << 16) + kACol + 32u * (uint32_t)s, unit, b, (row_t % 64) / 16, lane,
                          rg_valid);
          tc_fence_before();
        } else {
#pragma unroll
          for (int h = 0; h < RPW / 16; ++h) {
            const int row0 = row_t + 16 * h;
            const int rt = (row0 % 64) / 16;
            convert_tile<F>(sm.b[s], unit, b, rt, row0, lane, rg_valid, swz);
            if constexpr (F == kSpqr) {
              if (rg_valid) {
                __syncwarp();
                const int64_t u = (rg0 + rg_local) * a.KU + ui;
                const uint32_t e0 = soffs(rg_local, 4 * u), e1 = soffs(rg_local, 4 * u + 4);
                const bool staged = e1 > e0 && e1 - e0 <= (uint32_t)kOutCapTc;
                spqr_outliers_tile(sm.b[s], staged ? sm.out[p][slot(rg_local)] : nullptr, e0 & ~3u, a.ents,
                                   soffs(rg_local, 4 * u + rt), soffs(rg_local, 4 * u + rt + 1), b, row0, lane);
              }
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.ab_full[s]);
          if constexpr (CL) {
            // the same rows into the partner's tile (RPW rows of 128 bytes, whole swizzle atoms);
            // its stage is free: both CTAs' tensor cores have read k-block i - NST
            const uint32_t o = (uint32_t)row_t * 128u;
            bulk_s2s_cluster(mapa_shared(smem_u32(sm.b[s] + o), partner), sm.b[s] + o, RPW * 128u,
                             mapa_shared(smem_u32(&sm.ab_full[s]), partner));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.pk_empty[p]);
    }
    if constexpr (F != kW8) {
      // epilogue (first converter group): TMEM lane quadrant q = warp % 4 holds weight rows
      // 32q.., the two warps of a quadrant take one 128-token half each; a warp's store of one
      // token writes 32 consecutive outputs of Y's row
      const int q = warp & 3;
      const int mh = (warp - 2) / 4;
      const bool epi = warp - 2 < 8;  // the first eight converter warps, two per TMEM lane quadrant
      if (epi && ok && mbar_wait(&sm.acc_full, 0u, a.status)) {
        tc_fence_after();
        if constexpr (kRowsInLanes) {
          const int n = n_tile * kBN + 32 * q + lane;
#pragma unroll 1
          for (int cb = 0; cb < 128 / 32; ++cb) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 128u * mh + 32u * cb, r);
            const int m0 = m_tile * BM + 128 * mh + 32 * cb;
            if (n < a.N) {
              uint16_t* dst = a.Y + (int64_t)m0 * a.N + n;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (m0 + i < a.M) dst[(int64_t)i * a.N] = f2bf(__uint_as_float(r[i]));
            }
          }
        } else {
          // lanes are tokens: each lane writes 32 consecutive outputs of its token's row
          const int m = m_tile * BM + 128 * mh + 32 * q + lane;
#pragma unroll
          for (int cb = 0; cb < kBN / 32; ++cb) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 128u * mh + 32u * cb, r);
            // N is a multiple of 64 rows (the device image pads row groups), so a 32-column
            // slice is either fully inside or fully outside the output
            const int n = n_tile * kBN + 32 * cb;
            if (m < a.M && n + 32 <= a.N) {
              uint32_t pk16[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk16[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
              uint16_t* dst = a.Y + (int64_t)m * a.N + n;
#pragma unroll
              for (int v = 0; v < 4; ++v)
                reinterpret_cast<uint4*>(dst)[v] = make_uint4(pk16[4 * v], pk16[4 * v + 1], pk16[4 * v + 2], pk16[4 * v + 3]);
            }
          }
        }
      }
    }
  } else if constexpr (F == kW8) {
    // ------------------------------------------------------------------ exact int32 drain + epilogue
    // warps 10..17: TMEM lane quadrant q = warp % 4 (weight rows 32q..32q+31), token half
    // mh = (warp - 10) / 4 (accumulator columns 128 mh.., 16-bit high parts 256 + 64 mh..)
    pdl_wait();
    const int q = warp & 3;
    const int mh = (warp - 2 - NCONV) / 4;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t fcol = 128u * mh, hcol = 256u + 64u * mh;
    const int n = n_tile * kBN + 32 * q + lane;  // this lane's weight row
    const float swn = n < a.N ? a.sw[n] : 0.f;
    int nchunks = 1;  // the MMA issuer's chunking, replayed
    // whether the tile's blocks fit one exact chunk: the sum of all block bounds, the 256 drain
    // threads taking every 256th block, so the MMA issuer finds the answer ready at k-block
    // kChunkMin - 1 (one lane walking every 32nd block took longer than those 15 blocks)
    {
      long long part = 0;
#if QLIN_W8_PLAN_PAR
      for (int j = (warp - 2 - NCONV) * 32 + lane; j < nkb; j += 256) part += block_bound(kb[j], kw[j]);
#else
      if (warp == 2 + NCONV)
        for (int j = lane; j < nkb; j += 32) part += block_bound(kb[j], kw[j]);
#endif
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0 && part) atomicAdd(&sm.plan_sum, (unsigned long long)part);
      named_bar_sync(1, 256);  // the eight drain warps
    }
    const bool one_chunk = sm.plan_sum <= (unsigned long long)kExactSum;
    if (warp == 2 + NCONV && lane == 0) {  // the MMA issuer reads it at k-block kChunkMin - 1
      sm.plan_one = one_chunk ? 1 : 0;
      mbar_arrive(&sm.plan_full);
    }
    for (int i = 0, bound = 0; i < nkb && !one_chunk; ++i) {
      const int bi = block_bound(kb[i], kw[i]);
      if (i > 0 && bound + bi > kExactSum) {
        ++nchunks;
        bound = bi;
      } else {
        bound += bi;
      }
    }
    for (int c = 0; c < nchunks && ok; ++c) {
      if (!mbar_wait(&sm.ch_full[0], (uint32_t)c & 1u, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool last = c == nchunks - 1;
#pragma unroll 1
      for (int cb = 0; cb < 8; ++cb) {  // 16 tokens at a time
        uint32_t r[16], h[8];
        tmem_ld16(tmem + lane_base + fcol + 16u * cb, r);
        if (c > 0) {
          tmem_ld8(tmem + lane_base + hcol + 8u * cb, h);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) h[i] = 0u;
        }
        if (!last) {  // v = 2^16 hi + lo: hi into the high part, lo back into the accumulator
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int32_t v0 = __float2int_rn(__uint_as_float(r[2 * i]));
            const int32_t v1 = __float2int_rn(__uint_as_float(r[2 * i + 1]));
            const int32_t h0 = (int32_t)(int16_t)(h[i] & 0xFFFFu) + (v0 >> 16);
            const int32_t h1 = (int32_t)(int16_t)(h[i] >> 16) + (v1 >> 16);
            h[i] = ((uint32_t)h0 & 0xFFFFu) | ((uint32_t)h1 << 16);
            r[2 * i] = __float_as_uint((float)(v0 & 0xFFFF));
            r[2 * i + 1] = __float_as_uint((float)(v1 & 0xFFFF));
          }
          tmem_st16(tmem + lane_base + fcol + 16u * cb, r);
          tmem_st8(tmem + lane_base + hcol + 8u * cb, h);
          continue;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int32_t h0 = (int32_t)(int16_t)(h[i] & 0xFFFFu), h1 = (int32_t)(int16_t)(h[i] >> 16);
          r[2 * i] = (uint32_t)((int32_t)((uint32_t)h0 << 16) + __float2int_rn(__uint_as_float(r[2 * i])));
          r[2 * i + 1] = (uint32_t)((int32_t)((uint32_t)h1 << 16) + __float2int_rn(__uint_as_float(r[2 * i + 1])));
        }
        // columns are tokens m0 + i; a warp's store of one token writes 32 consecutive outputs
        const int m0 = m_tile * BM + 128 * mh + 16 * cb;
        if (n >= a.N) continue;
        if (a.acc_out) {
          int32_t* dst = a.acc_out + (int64_t)m0 * a.N + n;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (m0 + i < a.M) dst[(int64_t)i * a.N] = (int32_t)r[i];
        } else if (m0 + 16 <= a.M) {  // whole 16-token slice: token scales as 16-byte loads
          uint16_t* dst = a.Y + (int64_t)m0 * a.N + n;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(a.sx + m0) + v);
            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 4 * v + e;
              dst[(int64_t)i * a.N] = f2bf(__fmul_rn(__fmul_rn(__int2float_rn((int32_t)r[i]), sv[e]), swn));
            }
          }
        } else {
          uint16_t* dst = a.Y + (int64_t)m0 * a.N + n;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (m0 + i < a.M)
              dst[(int64_t)i * a.N] = f2bf(__fmul_rn(__fmul_rn(__int2float_rn((int32_t)r[i]), a.sx[m0 + i]), swn));
        }
      }
      if (!last) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.ch_empty[0]);
      }
    }
  }

  __syncwarp();
  // CL: neither CTA leaves while the partner may still write into its tile or barriers
  if constexpr (CL) cluster_sync_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

template <int F>
int launch_tc(const void* Xop, const TcArgs& args, void* stream) {
  using C = TcCfg<F>;
  constexpr int BM = 128 * C::kMH;
  if constexpr (F == kSpqr) {
    if (4 * (int64_t)args.KU + 8 > kOffsCapTc) return (int)cudaErrorInvalidValue;  // K > 65536: not staged
  }
  auto enc = tensor_map_encoder();
  if (!enc) return (int)cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)args.K, (cuuint64_t)args.M};
  const cuuint64_t strides[1] = {(cuuint64_t)args.K * 2};
  const cuuint32_t box[2] = {kBK, (cuuint32_t)BM};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = F == kW8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(&map, dt, 2, const_cast<void*>(Xop), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  const int mt_count = (args.M + BM - 1) / BM;
  // SpQR with an even number of token tiles: CTA pairs (every pair of consecutive tiles of the
  // grouped raster shares its weight tile then)
  const bool pair = F == kSpqr && QLIN_TC_SPQR_PAIRS && mt_count % 2 == 0;
  static_assert(sizeof(TcSmem<F, true>) + 1024 <= 227 * 1024 && sizeof(TcSmem<F>) + 1024 <= 227 * 1024,
                "shared memory per CTA");
  const size_t smem = (pair ? sizeof(TcSmem<F, true>) : sizeof(TcSmem<F>)) + 1024;
  auto* kern = pair ? tc_gemm_kernel<F, F == kSpqr> : tc_gemm_kernel<F, false>;
  static std::atomic<uint64_t> attr_done[2];
  if (const int e = smem_attr_once(kern, smem, attr_done[pair ? 1 : 0])) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((args.N + kBN - 1) / kBN) * mt_count));
  cfg.blockDim = dim3(tc_threads<F>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = QLIN_USE_PDL;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pair ? 2 : 1;
  return (int)cudaLaunchKernelEx(&cfg, kern, map, args);
}

}  // namespace

int launch_w4_prefill(const W4View& v, const uint16_t* X, uint16_t* Y, int M, int32_t* status, void* stream) {
  TcArgs a{v.units, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, Y, nullptr, status, M, v.N, v.K, v.RG, v.G};
  return launch_tc<kW4>(X, a, stream);
}

int launch_spqr_prefill(const SpqrView& v, const uint16_t* X, uint16_t* Y, int M, int32_t* status, void* stream) {
  TcArgs a{v.units, v.offs, v.ents, nullptr, nullptr, nullptr, nullptr, Y, nullptr, status, M, v.N, v.K, v.RG, v.S};
  return launch_tc<kSpqr>(X, a, stream);
}

int launch_w8_prefill(const W8View& v, const uint16_t* q16, const float* sx, const int32_t* kbound, uint16_t* Y,
                      int32_t* acc, int M,
                      int32_t* status, void* stream) {
  TcArgs a{v.units, nullptr, nullptr, v.sw, sx, kbound, v.w2, Y, acc, status, M, v.N, v.K, v.RG, v.KB};
  return launch_tc<kW8>(q16, a, stream);
}

}  // namespace qlin

// Single-token decode (M == 1) of the W4 g128 and SpQR formats: y = W_hat x, the layer's
// compressed weights streamed once.
//
// GPTQ page ("Makale Bülteni — GPTQ", "İddia ve Gerçeklik: GPTQ"): at batch one a
// weight-only 4-bit layer is bound by the bytes of its weights.  SpQR page ("Makale
// Bülteni — SpQR", "İddia ve Gerçeklik: SpQR"): the kernel unpacks the dense 3-bit codes
// and applies the sparse fp16 outliers in the same pass.
//
// Organisation (one launch per forward):
// * a CTA is two groups of four consumer warps, each with its producer warp.  A group is a
//   worker with its own contiguous range of units (64 rows x one K unit: a 128-wide group
//   for W4, a 256-wide supergroup for SpQR) and its own shared-memory ring, which its
//   producer fills with cp.async.bulk while it prefetches the units after the ring into L2
//   (the streamed copies are marked evict-first, so they do not push prefetched lines out);
// * two CTAs per SM (sixteen consumer warps keep the issue slots busy; the work is issue
//   bound); one for layers under 10 MB, whose start-up weighs more than their units.  Under programmatic dependent launch a CTA of the next forward issues its first
//   weight copies and L2 prefetches (weights never depend on the previous kernel) as soon as
//   a CTA of this one leaves its SM.  (Measured alternatives: one CTA of four groups, and one
//   co-resident CTA of two groups per forward, were as fast or slower.);
// * the token's activations are copied into shared memory once per CTA (the K units its
//   range touches, by a thread of their own right after griddepcontrol.wait, so the copy
//   never waits behind the weight stream's set-up) and the sums of x that the formulation
//   needs are prepared once per CTA, so a unit costs only its weight bytes.  The CTAs that
//   become resident only as the previous forward leaves set the forward's end: for them this
//   prologue is on the critical path;
// * integer-exact MMA formulation: the A operand is bf16(base + q) made from the code bits
//   with one AND/OR per register pair, (base + q) x accumulates in fp32, and the base and
//   zero-point terms come off once per (row, group) through the prepared sums of x.  A
//   one-hot x therefore reproduces bf16(w_hat) bit for bit;
// * SpQR outliers: the lanes of a warp take a bucket's entries round robin and add
//   value * x[k] into per-(row, lane) slots in shared memory; the flush of a row group sums
//   the slots in a fixed order (deterministic, no atomics, every lane busy however the
//   outliers fall over the rows);
// * a row group split between workers is finished by the worker holding its first unit:
//   the others store tagged partial words in the workspace and move on (no atomics), and
//   every wait is bounded in time.
#include "kern_decode_common.cuh"

namespace qlin {
namespace {

#ifndef QLIN_G1_GROUPS
#define QLIN_G1_GROUPS 2
#endif
#ifndef QLIN_G1_CTAS_PER_SM
#define QLIN_G1_CTAS_PER_SM 2
#endif
constexpr int kG1Groups = QLIN_G1_GROUPS;                     // workers per CTA
constexpr int kG1CtasPerSm = QLIN_G1_CTAS_PER_SM;             // CTAs of one forward per SM
constexpr int kG1Consumers = 4 * kG1Groups;                    // consumer warps
constexpr int kG1Threads = 32 * (kG1Consumers + kG1Groups);  // + one producer warp per group
constexpr int kG1MaxStages = 8;
#ifndef QLIN_G1_SP_STAGES
#define QLIN_G1_SP_STAGES 3
#endif
#ifndef QLIN_G1_W4_STAGES
#define QLIN_G1_W4_STAGES 4
#endif
constexpr int kG1SpStages = QLIN_G1_SP_STAGES;  // ring depth per group (one less if it does not fit)
constexpr int kG1W4Stages = QLIN_G1_W4_STAGES;
// units a producer prefetches into L2 ahead of its shared-memory ring: with the ring this
// keeps about 100 KB per group in flight from DRAM, and the co-resident next forward's
// producers pull that much of their own layer into L2 before griddepcontrol.wait returns
#ifndef QLIN_G1_PREFETCH
#define QLIN_G1_PREFETCH 1
#endif
constexpr int kG1SpPrefetch = QLIN_G1_PREFETCH ? 12 : 0;
constexpr int kG1W4Prefetch = QLIN_G1_PREFETCH ? 24 : 0;
constexpr uint32_t kG1WaitHintNs = 20000;  // suspend-time hint of a consumer's barrier poll
constexpr int kG1OutCap = 504;    // outlier entries staged with a unit (more: read from global)
constexpr int kG1OutWords = 512;  // words of a stage's outlier area (the copy is 16-byte aligned)
constexpr int kG1OffsCap = 2048;  // staged bucket offsets per CTA: ranges of at most 511 units
constexpr int kG1MaxUnitsPerCta = kG1OffsCap / 4 - 1;
constexpr size_t kG1MaxSmem = 227 * 1024;  // dynamic shared memory limit of a CTA

struct G1Hdr {
  uint64_t full[kG1Groups][kG1MaxStages];
  uint64_t empty[kG1Groups][kG1MaxStages];
  uint64_t grp_bar[kG1Groups];  // the four warps of a group (128 arrivals)
  uint64_t all_bar;             // every consumer thread
  uint64_t x_bar;               // the staged activations (transaction count)
  uint64_t offs_bar;            // the staged bucket offsets (SpQR)
  uint64_t perm_bar;            // the staged permutation entries (W4 act-order)
  int64_t u0[kG1Groups + 1];    // unit ranges: group g owns [u0[g], u0[g + 1])
  int64_t rg0[kG1Groups];       // row group of each group's first unit
  int k0[kG1Groups];            // K unit (within the row) of each group's first unit
  int ls0[kG1Groups];           // and its index in the staged activations
  int rg[kG1Groups][2];         // row groups shared with other workers: first / last of the range
  int owned[kG1Groups];         // side of the shared row group this worker finishes (-1: none)
  int others[kG1Groups];        // workers after this one that contribute to it
  int xn;                       // K units of x staged
  int pad_;
  float own[kG1Groups][kRowGroup];  // the finishing worker's own sums of its shared row group
  __align__(16) uint32_t zeros[16];
};

}  // namespace

// Section offsets of the dynamic shared memory (from the 128-byte aligned base)
// floor(n / d) by a multiply with a precomputed inverse of d, for every 32-bit n (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994, Figure 4.1)
struct G1Div {
  uint32_t m, s1, s2;
};

struct G1Layout {
  uint32_t ring;         // [groups][stages] stages of stage_bytes
  uint32_t stage_bytes;
  uint32_t offs;         // SpQR: staged bucket offsets
  uint32_t slots;        // SpQR: outlier slots [consumer warps][16 rows][32 lanes] fp32
  uint32_t gtab;         // sums of x per group of the staged K units
  uint32_t xs;           // staged x, plain order
  uint32_t xf;           // W4: staged x in B-fragment order
  uint32_t bytes;        // total
  uint32_t xfull;        // W4 act-order: the whole x row (input channel order)
  uint32_t perm;         // W4 act-order: the permutation entries of the staged K units
  G1Div dW, dU, dR;      // inverses of the worker count, the unit count and the units per row group
};

namespace {

inline uint32_t al128(uint32_t x) { return (x + 127u) & ~127u; }

G1Layout g1_layout(bool spqr, int xn, int stages, int xfull_k = 0) {
  G1Layout L{};
  uint32_t o = al128((uint32_t)sizeof(G1Hdr));
  L.stage_bytes = spqr ? al128(kSpqrUnitBytes + kG1OutWords * 4) : al128(kW4UnitBytes);
  L.ring = o;
  o += L.stage_bytes * kG1Groups * stages;
  if (spqr) {
    L.offs = o;
    o = al128(o + kG1OffsCap * 4);
    L.slots = o;
    o = al128(o + kG1Consumers * 16 * 32 * 4);
    L.gtab = o;  // [xn][2 blocks][4 t]: float4 (-B(2t), -B(2t+1), -B(2t), -B(2t+1)), then float2 (S(2t), S(2t+1))
    o = al128(o + (uint32_t)xn * 8 * (16 + 8));
    L.xs = o;
    o = al128(o + (uint32_t)xn * kSpqrSuper * 2);
  } else {
    L.gtab = o;
    o = al128(o + (uint32_t)xn * 4);
    L.xs = o;
    o = al128(o + (uint32_t)xn * kW4Group * 2);
    L.xf = o;
    o = al128(o + (uint32_t)xn * kW4Group * 2);
    L.xfull = o;  // act-order: the whole token, in input channel order
    o = al128(o + (uint32_t)xfull_k * 2);
    L.perm = o;
    o = al128(o + (xfull_k ? (uint32_t)xn * kW4Group * 4 : 0u));
  }
  L.bytes = o;
  return L;
}

G1Div g1_div_make(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < d) ++l;  // ceil(log2 d)
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
  return {(uint32_t)m, l < 1 ? l : 1u, l > 1 ? l - 1 : 0u};
}

// floor(a / b) of non-negative a and b, v the inverse of b: a high multiply and two shifts
// when a fits 32 bits (every realistic layer).  The plan's chains of divisions are on the
// critical path of every CTA that starts late; done by the division routine they took about
// a microsecond.
__device__ __forceinline__ int64_t g1_div(int64_t a, int64_t b, const G1Div& v) {
  if ((uint64_t)a >> 32) return a / b;
  const uint32_t n = (uint32_t)a, t1 = __umulhi(n, v.m);
  return (int64_t)((t1 + ((n - t1) >> v.s1)) >> v.s2);
}

// Work plan of a CTA, computed by warp 0: its workers' unit ranges, where their ranges
// share row groups with other workers, and the K units of x the CTA needs.  Worker w owns
// units [w U / W, (w + 1) U / W); the owner of unit u is ((u + 1) W - 1) / U.
__device__ void g1_plan_warp(G1Hdr& h, int64_t U, int64_t per_rg, int lane, const G1Layout& L) {
  const int64_t W = (int64_t)gridDim.x * kG1Groups, c0 = (int64_t)blockIdx.x * kG1Groups;
  if (lane <= kG1Groups) h.u0[lane] = g1_div((c0 + lane) * U, W, L.dW);
  __syncwarp();
  const int64_t u0c = h.u0[0];
  if (lane < kG1Groups) {
    const int64_t u0 = h.u0[lane], rg0 = g1_div(u0, per_rg, L.dR), d = u0 - u0c;
    h.rg0[lane] = rg0;
    h.k0[lane] = (int)(u0 - rg0 * per_rg);
    h.ls0[lane] = (int)(d - g1_div(d, per_rg, L.dR) * per_rg);
    h.owned[lane] = -1;
    h.others[lane] = 0;
  }
  if (lane == 0) {
    const int64_t n = h.u0[kG1Groups] - u0c;
    h.xn = (int)(n < per_rg ? n : per_rg);
  }
  __syncwarp();
  if (lane < 2 * kG1Groups) {
    const int g = lane >> 1, s = lane & 1;
    const int64_t w = c0 + g, u0 = h.u0[g], u1 = h.u0[g + 1];
    int out = -1;
    if (u1 > u0) {
      const int64_t r = g1_div(s == 0 ? u0 : u1 - 1, per_rg, L.dR);
      if (!(s == 1 && r == h.rg0[g])) {
        const int64_t first = g1_div((r * per_rg + 1) * W - 1, U, L.dU);
        const int64_t last = g1_div((r * per_rg + per_rg) * W - 1, U, L.dU);
        if (first != last) {
          out = (int)r;
          if (first == w) {  // at most one side: a range starting at its row group's first unit
            h.owned[g] = s;   // and ending inside it has no second row group
            h.others[g] = (int)(last - first);
          }
        }
      }
    } else if (s == 0 && u0 < U) {
      // an empty range (more workers than units) that sits inside a shared row group still
      // counts among its contributors: it contributes zeros
      const int64_t r = g1_div(u0, per_rg, L.dR);
      const int64_t first = g1_div((r * per_rg + 1) * W - 1, U, L.dU);
      const int64_t last = g1_div((r * per_rg + per_rg) * W - 1, U, L.dU);
      if (first < w && w <= last) out = (int)r;
    }
    h.rg[g][s] = out;
  }
}

// Bounded barrier wait that suspends between polls (a waiting consumer issues almost nothing)
__device__ __forceinline__ bool g1_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, kG1WaitHintNs)) return true;
    if (global_ns() - t0 > kWaitLimitNs) break;
  }
  atomicExch(status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// L2 policy for data read once (the weight stream): first to be evicted after the read
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void bulk_g2s_ef(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// L2 prefetch of a 16-byte aligned range (size a multiple of 16), in pieces of at most 32 KB
__device__ __forceinline__ void prefetch_l2(const void* src, uint64_t bytes) {
  const char* p = static_cast<const char*>(src);
  while (bytes > 0) {
    const uint32_t b = bytes > 32768 ? 32768u : (uint32_t)bytes;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(b) : "memory");
    p += b;
    bytes -= b;
  }
}

// Completion of a worker's row groups (one token).  stage(): a row group the worker holds
// whole goes to `done`; a shared one goes to shared memory (the worker finishes it) or, as
// a tagged 8-byte word, to the worker's slot in the workspace.  finish(): the finishing
// worker waits (bounded) for the other contributors' words, adds them in worker order and
// clears them, so no slot holds a valid-looking word between forwards.
struct G1Fin {
  uint64_t* tagged;
  float* own;
  int32_t* status;
  uint32_t tag;
  int w;
  int rg0, rg1, owned, others;

  __device__ __forceinline__ uint64_t* slot(int c, int side) const {
    return tagged + (int64_t)(c * 2 + side) * (kRowGroup * 4);
  }

  template <typename Done>
  __device__ __forceinline__ void stage(int64_t r, int row, float val, Done done) const {
    const int s = (r == rg0) ? 0 : (r == rg1) ? 1 : -1;
    if (s < 0) {
      done(r, row, val);
    } else if (s == owned) {
      own[row] = val;
    } else {
      st_relaxed_b64(slot(w, s) + row, ((uint64_t)tag << 32) | __float_as_uint(val));
    }
  }

  // gtid: thread index within the group (0..127); the group barrier orders the own[] stores
  template <typename Put>
  __device__ __forceinline__ bool finish(ConsumerSync& cs, int gtid, Put put) const {
    if (owned < 0) return true;
    if (!cs.sync()) return false;
    if (gtid >= kRowGroup) return true;
    const int row = gtid;
    float acc = own[row];
    constexpr int B = 8;  // contributors loaded per L2 round trip
    for (int c0 = 0; c0 < others; c0 += B) {
      uint64_t vv[B];
#pragma unroll
      for (int u = 0; u < B; ++u) vv[u] = (c0 + u < others) ? ld_relaxed_b64(slot(w + 1 + c0 + u, 0) + row) : 0ull;
      uint64_t t0 = 0;
      for (;;) {
        unsigned missing = 0;
#pragma unroll
        for (int u = 0; u < B; ++u)
          if (c0 + u < others && (uint32_t)(vv[u] >> 32) != tag) missing |= 1u << u;
        if (!missing) break;
        if (t0 == 0) {
          t0 = global_ns();
        } else if (global_ns() - t0 > kWaitLimitNs) {
          atomicExch(status, kStatusTimeout);
          return false;
        }
#pragma unroll
        for (int u = 0; u < B; ++u)
          if (missing & (1u << u)) vv[u] = ld_relaxed_b64(slot(w + 1 + c0 + u, 0) + row);
      }
#pragma unroll
      for (int u = 0; u < B; ++u) {
        if (c0 + u >= others) continue;
        acc += __uint_as_float((uint32_t)vv[u]);
        st_relaxed_b64(slot(w + 1 + c0 + u, 0) + row, 0ull);
      }
    }
    put((int64_t)(owned == 0 ? rg0 : rg1), row, acc);
    return true;
  }
};

__device__ __forceinline__ float2 h2f2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& p, float (&e)[8]) {
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    e[2 * i] = __uint_as_float(w[i] << 16);
    e[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// D = A * B + C with C in other registers than D (fp32 accumulate, bf16 operands)
__device__ __forceinline__ void mma_bf16_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                           const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

__device__ __forceinline__ void mma_bf16_c4(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                            const float4& c) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}

// Shared-memory accesses by 32-bit shared address
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// One SpQR outlier entry (fp16 value << 16 | k in the 256-wide unit << 4 | row in the tile):
// slot[row][lane] += value * x[k].  slot_lane: this lane's slot of row 0 (rows 128 bytes apart);
// xsg: the unit's 256 staged activations (bf16).
__device__ __forceinline__ void slot_add(uint32_t slot_lane, uint32_t e, uint32_t xsg) {
  const uint32_t sa = slot_lane + ((e & 15u) << 7);
  const float x = __uint_as_float(lds_u16(xsg + ((e >> 3) & 0x1FEu)) << 16);
  const float val = __half2float(__ushort_as_half((uint16_t)(e >> 16)));
  sts_f32(sa, fmaf(val, x, lds_f32(sa)));
}

// ---------------------------------------------------------------------------------- SpQR

// (a & MASK) | c as one LOP3: the mask is the instruction's immediate and c a register
// (a constant OR-ed after a mask would otherwise cost a second logic instruction)
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}

// bf16 exponent patterns the code fields are OR-ed under: 128 + q (fields at bits 0..2 of
// a half) and 16 + q (fields at bits 3..5), held in registers
struct SpOr {
  uint32_t b128, b16;
};

// A register pair for MMA j, register r, from the lane's six code words of a block (the
// field layout of the device image: bf16 128 + q for MMA 0..4, 16 + q for MMA 5..7)
template <int J, int R>
__device__ __forceinline__ uint32_t sp_pair(const uint32_t (&w)[6], const SpOr& k) {
  if constexpr (J <= 4) {
    constexpr int i = 4 * J + R;
    if constexpr (i < 18) {
      constexpr int wi = i / 3, f = (i % 3) * 2;
      return and_or<0x00070007u>(w[wi] >> (3 * f), k.b128);
    } else {
      // the three spare bits (15 and 31) of three consecutive words
      constexpr int b = 3 * (i - 18);
      const uint32_t p = and_or<0x00010001u>(w[b] >> 15, k.b128);
      const uint32_t q = and_or<0x00020002u>(w[b + 1] >> 14, p);
      return and_or<0x00040004u>(w[b + 2] >> 13, q);
    }
  } else {
    constexpr int i = 4 * (J - 5) + R;
    constexpr int wi = i / 2, f = (i % 2) * 2 + 1;
    return and_or<0x00380038u>(w[wi] >> (3 * (f - 1)), k.b16);
  }
}

// One MMA of the block-diagonal product, regrouped so that both k halves of the MMA belong
// to one 16-group: MMA m of set h (h = 0: groups 0..3 of the block, h = 1: groups 4..7)
// takes, for the lane's group t + 4h, elements 4m, 4m + 1 (k columns 2t, 2t + 1) and 4m + 2,
// 4m + 3 (columns 2t + 8, 2t + 9) -- the pairs that the device layout keeps in register r
// = 2h, 2h + 1 of its MMAs 2m and 2m + 1.  The B operand of column g then holds four
// consecutive activations of group g (one aligned register pair) on the four lanes of the
// set's diagonal and zeros elsewhere, and accumulator column n still sums group n.
template <int M, int H, bool Z = false>
__device__ __forceinline__ void sp_mma(const uint32_t (&w)[6], const SpOr& k, const uint32_t (&b)[8],
                                       float (&c)[4]) {
  uint32_t a[4];
  a[0] = sp_pair<2 * M, 2 * H>(w, k);
  a[1] = sp_pair<2 * M, 2 * H + 1>(w, k);
  a[2] = sp_pair<2 * M + 1, 2 * H>(w, k);
  a[3] = sp_pair<2 * M + 1, 2 * H + 1>(w, k);
  if constexpr (Z) {  // the first MMA of a chain: zero C operand
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16_c(c, a, b[2 * M], b[2 * M + 1], zero4);
  } else {
    mma_bf16(c, a, b[2 * M], b[2 * M + 1]);
  }
}

template <int STAGES>
__global__ void __launch_bounds__(kG1Threads, kG1CtasPerSm)
    spqr_gemv1_kernel(SpqrView v, const uint16_t* __restrict__ X, uint16_t* __restrict__ Y, Workspace ws,
                      G1Layout L) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* sb = smem_align128(smem_raw);
  G1Hdr& h = *reinterpret_cast<G1Hdr*>(sb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t S = v.S, U = (int64_t)v.RG * S, vN = v.N;
  uint32_t* offs_s = reinterpret_cast<uint32_t*>(sb + L.offs);
  float* slots = reinterpret_cast<float*>(sb + L.slots);
  float4* gq = reinterpret_cast<float4*>(sb + L.gtab);
  uint16_t* xs = reinterpret_cast<uint16_t*>(sb + L.xs);
  const int g = lane >> 2, t = lane & 3;

  if (warp == 0) g1_plan_warp(h, U, S, lane, L);
  if (threadIdx.x == 32) {
#pragma unroll
    for (int q = 0; q < kG1Groups; ++q) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&h.full[q][s], 1);
        mbar_init(&h.empty[q][s], 128);  // every consumer thread of the group releases
      }
      mbar_init(&h.grp_bar[q], 128);
    }
    mbar_init(&h.all_bar, 32 * kG1Consumers);
    mbar_init(&h.x_bar, 1);
    mbar_init(&h.offs_bar, 1);
    fence_mbar_init();
    pdl_launch_dependents();
    // Weights never depend on the previous kernel: the CTA's bucket offsets and each group's
    // first ring units go out now, before the plan is shared (the same unit ranges as the
    // plan's).  A CTA that becomes resident only when the previous forward's CTAs leave its SM
    // has its first units' outliers on the critical path, behind the offsets' round trip:
    // issuing that here took the 11008 x 4096 forward from 10.3 to 9.6 us.  (W4, with no such
    // round trip, is faster with its producers issuing after the plan.)
    int64_t ub[kG1Groups + 1];
    const int64_t W = (int64_t)gridDim.x * kG1Groups, c0 = (int64_t)blockIdx.x * kG1Groups;
#pragma unroll
    for (int q = 0; q <= kG1Groups; ++q) ub[q] = g1_div((c0 + q) * U, W, L.dW);
    if (ub[kG1Groups] > ub[0]) {
      const int64_t ob = 4 * ub[0], oe = 4 * ub[kG1Groups] + 4;
      mbar_arrive_expect_tx(&h.offs_bar, (uint32_t)(oe - ob) * 4u);
      bulk_g2s(offs_s, v.offs + ob, (uint32_t)(oe - ob) * 4u, &h.offs_bar);
      const uint64_t pol = policy_evict_first();
#pragma unroll
      for (int q = 0; q < kG1Groups; ++q) {
        const int n = (int)(ub[q + 1] - ub[q]);
        for (int i = 0; i < (n < STAGES ? n : STAGES); ++i) {  // completed by the outliers' arrival
          mbar_expect_tx(&h.full[q][i], kSpqrUnitBytes);
          bulk_g2s_ef(sb + L.ring + (uint32_t)(q * STAGES + i) * L.stage_bytes,
                      v.units + (ub[q] + i) * (int64_t)kSpqrUnitBytes, kSpqrUnitBytes, &h.full[q][i], pol);
        }
      }
    }
  }
  if (threadIdx.x >= 64 && threadIdx.x < 80) h.zeros[threadIdx.x - 64] = 0u;
  if (warp < kG1Consumers) {
    // every lane clears the outlier slots it sums at a flush: rows g and g + 8, lanes 8t..8t+7
    float4* sl = reinterpret_cast<float4*>(slots + warp * 512);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    sl[(g * 32 + 8 * t) / 4] = z4;
    sl[(g * 32 + 8 * t) / 4 + 1] = z4;
    sl[((g + 8) * 32 + 8 * t) / 4] = z4;
    sl[((g + 8) * 32 + 8 * t) / 4 + 1] = z4;
  }
  __syncthreads();
  const int64_t u0c = h.u0[0], u1c = h.u0[kG1Groups];
  if (u1c <= u0c) return;  // no units for this CTA (uniform)

  if (warp >= kG1Consumers) {
    // ------------------------------------------- producers: one thread per group, own ring
    const int q = warp - kG1Consumers;
    if (q == 0 && lane == 1) {
      // x, as soon as the previous kernel is done (apart from the weight stream, which may
      // still wait for its bucket offsets)
      pdl_wait();  // x is written by the previous kernel on the stream
      const int xn = h.xn;
      const int64_t ks = u0c - g1_div(u0c, S, L.dR) * S;
      const int na = (int)((int64_t)xn < S - ks ? (int64_t)xn : S - ks);
      mbar_arrive_expect_tx(&h.x_bar, (uint32_t)xn * (kSpqrSuper * 2));
      bulk_g2s(xs, X + ks * kSpqrSuper, (uint32_t)na * (kSpqrSuper * 2), &h.x_bar);
      if (xn > na) bulk_g2s(xs + (size_t)na * kSpqrSuper, X, (uint32_t)(xn - na) * (kSpqrSuper * 2), &h.x_bar);
      return;
    }
    if (lane != 0) return;
    const int64_t a = h.u0[q];
    const int n = (int)(h.u0[q + 1] - a);
    const uint64_t pol = policy_evict_first();
    auto stage_at = [&](int s) { return sb + L.ring + (uint32_t)(q * STAGES + s) * L.stage_bytes; };
    auto unit_src = [&](int i) { return v.units + (a + i) * (int64_t)kSpqrUnitBytes; };
    // outlier entries of unit a + i staged with it (16-byte aligned range), or none
    auto out_range = [&](int i, uint32_t& a0, uint32_t& a1) {
      const int oi = 4 * (int)(a + i - u0c);
      const uint32_t e0 = offs_s[oi], e1 = offs_s[oi + 4];
      a0 = e0 & ~3u;
      a1 = (e1 + 3u) & ~3u;
      return e1 > e0 && e1 - e0 <= (uint32_t)kG1OutCap;
    };
    auto prefetch = [&](int i0, int i1) {  // units [i0, i1) and their outliers into L2
      if (i1 <= i0) return;
      prefetch_l2(unit_src(i0), (uint64_t)(i1 - i0) * kSpqrUnitBytes);
      const uint32_t e0 = offs_s[4 * (int)(a + i0 - u0c)] & ~3u, e1 = (offs_s[4 * (int)(a + i1 - u0c)] + 3u) & ~3u;
      if (e1 > e0) prefetch_l2(v.ents + e0, (uint64_t)(e1 - e0) * 4u);
    };
    // the ring's first units went out with the barrier set-up; their outliers follow once the
    // offsets are in
    const int pro = n < STAGES ? n : STAGES;
    if (!mbar_wait(&h.offs_bar, 0, ws.status)) return;
    for (int i = 0; i < pro; ++i) {
      uint32_t a0, a1;
      const bool so = out_range(i, a0, a1);
      mbar_arrive_expect_tx(&h.full[q][i], so ? (a1 - a0) * 4u : 0u);
      if (so) bulk_g2s_ef(stage_at(i) + kSpqrUnitBytes, v.ents + a0, (a1 - a0) * 4u, &h.full[q][i], pol);
    }
    int pf = pro + kG1SpPrefetch < n ? pro + kG1SpPrefetch : n;  // end of the prefetched window
    prefetch(pro, pf);
    int s = 0;
    uint32_t ph = 1u;  // the ring's first pass is done: waiting for the consumers' first release
    for (int i = pro; i < n; ++i) {
      if (!g1_wait(&h.empty[q][s], ph ^ 1u, ws.status)) return;
      uint32_t a0, a1;
      const bool so = out_range(i, a0, a1);
      mbar_arrive_expect_tx(&h.full[q][s], kSpqrUnitBytes + (so ? (a1 - a0) * 4u : 0u));
      bulk_g2s_ef(stage_at(s), unit_src(i), kSpqrUnitBytes, &h.full[q][s], pol);
      if (so) bulk_g2s_ef(stage_at(s) + kSpqrUnitBytes, v.ents + a0, (a1 - a0) * 4u, &h.full[q][s], pol);
      if (pf < n) {
        prefetch(pf, pf + 1);
        ++pf;
      }
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int grp = warp >> 2, rt = warp & 3;
  pdl_wait();  // workspace words and Y are touched only after the previous kernel is done
  if (!g1_wait(&h.x_bar, 0, ws.status)) return;
  // per 16-group of the staged x: -(sum of base * x) (base 128 for elements 0..9, 16 for
  // 10..15, as the code fields) and sum x, stored per (K unit, block, accumulator column
  // pair) as the C operand quad of the first MMA and the pair of sums
  float2* gs = reinterpret_cast<float2*>(gq + h.xn * 8);
  for (int w = threadIdx.x; w < h.xn * 8; w += 32 * kG1Consumers) {
    float nb[2], sm[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int lg = (w >> 2) * 8 + 2 * (w & 3) + c;  // 16-group in the staged x
      float e[8], f[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(xs + lg * 16), e);
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(xs + lg * 16 + 8), f);
      const float s128 = (((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]))) + (f[0] + f[1]);
      const float s16 = ((f[2] + f[3]) + (f[4] + f[5])) + (f[6] + f[7]);
      nb[c] = -(128.f * s128 + 16.f * s16);
      sm[c] = s128 + s16;
    }
    gq[w] = make_float4(nb[0], nb[1], nb[0], nb[1]);
    gs[w] = make_float2(sm[0], sm[1]);
  }
  mbar_arrive(&h.all_bar);
  if (!g1_wait(&h.all_bar, 0, ws.status)) return;

  const int64_t u0 = h.u0[grp];
  const int n_units = (int)(h.u0[grp + 1] - u0);
  const G1Fin fin{ws.tagged, h.own[grp], ws.status, ws.tag, (int)(blockIdx.x * kG1Groups + grp),
                  h.rg[grp][0], h.rg[grp][1], h.owned[grp], h.others[grp]};
  ConsumerSync cs{&h.grp_bar[grp], 0u, ws.status};
  float* myslots = slots + warp * 512;
  auto done = [&](int64_t r, int row, float val) {
    const int64_t nrow = r * kRowGroup + row;
    if (nrow < vN) Y[nrow] = f2bf(val);
  };
  // B operands: the block-diagonal activation matrix.  Lane (g, t) supplies column g: for the
  // MMAs of set 0 group g of the block when g == t, for set 1 group g when g == t + 4, zeros
  // otherwise (read from a zero area, which a step of 0 keeps them on).
  const bool d0 = g == t, d1 = g == t + 4;
  const uint8_t* zb = reinterpret_cast<const uint8_t*>(h.zeros);
  const uint8_t* xb0 = d0 ? reinterpret_cast<const uint8_t*>(xs) + 32 * g : zb;
  const uint8_t* xb1 = d1 ? reinterpret_cast<const uint8_t*>(xs) + 32 * g : zb;
  const int xst0 = d0 ? kSpqrSuper * 2 : 0, xst1 = d1 ? kSpqrSuper * 2 : 0;  // bytes per staged K unit
  const int xbk0 = d0 ? 256 : 0, xbk1 = d1 ? 256 : 0;                      // block 1 of the unit
  // this lane's offsets inside a stage
  const uint8_t* ring = sb + L.ring + (uint32_t)(grp * STAGES) * L.stage_bytes;
  const int code_off = ((rt * 2) * 32 + lane) * 24;  // block 1 at + 32 * 24
  const int stat_off = kSpqrCodeBytes + kSpqrQsqzBytes + (rt * 16 + g) * 8;  // row g + 8 at + 64
  const int qsqz_word = (24 * lane) >> 5, qsqz_sh = (24 * lane) & 31;
  const int qsqz_off = kSpqrCodeBytes + (rt * 2) * 96;  // block 1 at + 96
  SpOr kor{0x43004300u, 0x41804180u};
  uint32_t kmagic = 0x4B000000u;
  const uint32_t slot_lane = smem_u32(myslots) + 4u * lane;  // slot of (row 0, this lane)
  const uint32_t xs_addr = smem_u32(xs);

  int64_t cur_rg = h.rg0[grp];
  int kq = h.k0[grp], ls = h.ls0[grp], s = 0;
  uint32_t ph = 0;
  int it = 0;
  while (it < n_units) {
    // the units of one row group, then its flush
    const int seg_end = it + (int)S - kq < n_units ? it + (int)S - kq : n_units;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (; it < seg_end; ++it) {
      if (!g1_wait(&h.full[grp][s], ph, ws.status)) return;
      const uint8_t* unit = ring + s * L.stage_bytes;
      // outliers of this row tile in this unit first (they are read from the stage): entry i
      // goes to lane i % 32, which adds value * x[k] into its slot of the entry's row
      {
        const uint32_t xsg = xs_addr + (uint32_t)ls * (kSpqrSuper * 2);
        const uint32_t* ob = offs_s + 4 * (it + (int)(u0 - u0c));
        const uint32_t e0 = ob[0], e1 = ob[4], b0 = ob[rt], b1 = ob[rt + 1];
        const int n = (int)(b1 - b0);
        if (n > 0) {  // warp-uniform
          if (e1 - e0 <= (uint32_t)kG1OutCap) {
            // staged with the unit: two entries per lane per pass
            const uint32_t eb = smem_u32(unit + kSpqrUnitBytes) + 4u * (b0 - (e0 & ~3u));
            for (int i = lane; i < n; i += 64) {
              const bool two = i + 32 < n;
              const uint32_t ea = lds_u32(eb + 4u * i);
              const uint32_t ec = two ? lds_u32(eb + 4u * (i + 32)) : 0u;
              slot_add(slot_lane, ea, xsg);
              if (two) slot_add(slot_lane, ec, xsg);
            }
          } else {
            const uint32_t* bg = v.ents + b0;
            for (int i = lane; i < n; i += 32) slot_add(slot_lane, __ldg(bg + i), xsg);
          }
        }
      }
      // the rest of the stage into registers, then the stage goes back to the producer:
      // second-level statistics of rows g and g + 8 ((ss, zs), (sz, zz)), the code words of
      // both blocks, and the lane's 24-bit (qs, qz) fields
      const uint2 stA = *reinterpret_cast<const uint2*>(unit + stat_off);
      const uint2 stB = *reinterpret_cast<const uint2*>(unit + stat_off + 64);
      uint32_t w0[6], w1[6];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const uint2 p = *reinterpret_cast<const uint2*>(unit + code_off + 8 * i);
        const uint2 q = *reinterpret_cast<const uint2*>(unit + code_off + 32 * 24 + 8 * i);
        w0[2 * i] = p.x;
        w0[2 * i + 1] = p.y;
        w1[2 * i] = q.x;
        w1[2 * i + 1] = q.y;
      }
      uint32_t f24[2];
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(unit + qsqz_off + blk * 96);
        f24[blk] = __funnelshift_r(qw[qsqz_word], qw[qsqz_word + 1], qsqz_sh);
      }
      mbar_arrive(&h.empty[grp][s]);  // this thread is done with the stage
      // sums of x of the accumulator columns 2t, 2t + 1 of both blocks
      const float4 qA = gq[ls * 8 + t], qB = gq[ls * 8 + 4 + t];
      const float2 gA = gs[ls * 8 + t], gB = gs[ls * 8 + 4 + t];
      float c0[4], c1[4], e0[4], e1[4];
      {
        uint32_t bx0[8], by0[8], bx1[8], by1[8];
        {
          const uint8_t* px = xb0 + ls * xst0;
          const uint8_t* py = xb1 + ls * xst1;
          const uint4 x0 = *reinterpret_cast<const uint4*>(px), x1 = *reinterpret_cast<const uint4*>(px + 16);
          const uint4 y0 = *reinterpret_cast<const uint4*>(py), y1 = *reinterpret_cast<const uint4*>(py + 16);
          const uint4 x2 = *reinterpret_cast<const uint4*>(px + xbk0);
          const uint4 x3 = *reinterpret_cast<const uint4*>(px + xbk0 + 16);
          const uint4 y2 = *reinterpret_cast<const uint4*>(py + xbk1);
          const uint4 y3 = *reinterpret_cast<const uint4*>(py + xbk1 + 16);
          bx0[0] = x0.x; bx0[1] = x0.y; bx0[2] = x0.z; bx0[3] = x0.w;
          bx0[4] = x1.x; bx0[5] = x1.y; bx0[6] = x1.z; bx0[7] = x1.w;
          by0[0] = y0.x; by0[1] = y0.y; by0[2] = y0.z; by0[3] = y0.w;
          by0[4] = y1.x; by0[5] = y1.y; by0[6] = y1.z; by0[7] = y1.w;
          bx1[0] = x2.x; bx1[1] = x2.y; bx1[2] = x2.z; bx1[3] = x2.w;
          bx1[4] = x3.x; bx1[5] = x3.y; bx1[6] = x3.z; bx1[7] = x3.w;
          by1[0] = y2.x; by1[1] = y2.y; by1[2] = y2.z; by1[3] = y2.w;
          by1[4] = y3.x; by1[5] = y3.y; by1[6] = y3.z; by1[7] = y3.w;
        }
        // the first MMA of each block adds the base term, so each chain ends at
        // sum_k (q_k x_k) over the (row, group) of the accumulator; the two blocks are two
        // independent chains
        {
          uint32_t a[4];
          a[0] = sp_pair<0, 0>(w0, kor);
          a[1] = sp_pair<0, 1>(w0, kor);
          a[2] = sp_pair<1, 0>(w0, kor);
          a[3] = sp_pair<1, 1>(w0, kor);
          mma_bf16_c4(c0, a, bx0[0], bx0[1], qA);
          a[0] = sp_pair<0, 0>(w1, kor);
          a[1] = sp_pair<0, 1>(w1, kor);
          a[2] = sp_pair<1, 0>(w1, kor);
          a[3] = sp_pair<1, 1>(w1, kor);
          mma_bf16_c4(c1, a, bx1[0], bx1[1], qB);
        }
        // the second set of each block in chains of its own (four chains of four MMAs)
        sp_mma<0, 1, true>(w0, kor, by0, e0);
        sp_mma<0, 1, true>(w1, kor, by1, e1);
        sp_mma<1, 0>(w0, kor, bx0, c0);
        sp_mma<1, 0>(w1, kor, bx1, c1);
        sp_mma<1, 1>(w0, kor, by0, e0);
        sp_mma<1, 1>(w1, kor, by1, e1);
        sp_mma<2, 0>(w0, kor, bx0, c0);
        sp_mma<2, 0>(w1, kor, bx1, c1);
        sp_mma<2, 1>(w0, kor, by0, e0);
        sp_mma<2, 1>(w1, kor, by1, e1);
        sp_mma<3, 0>(w0, kor, bx0, c0);
        sp_mma<3, 0>(w1, kor, bx1, c1);
        sp_mma<3, 1>(w0, kor, by0, e0);
        sp_mma<3, 1>(w1, kor, by1, e1);
      }
      // first-level statistics of the accumulator's (row, group) pairs, decoded exactly:
      // a 3-bit field at bit p OR-ed under the exponent of 2^23 is the float 2^23 + q 2^p;
      // subtracting 2^23 + z 2^p and scaling by s 2^-p gives (q - z) s with one rounding
      {
        const float2 sA = h2f2(stA.x), zA = h2f2(stA.y), sB = h2f2(stB.x), zB = h2f2(stB.y);
        float kcs[4], kms[4], kcz[4], kmz[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float P = (float)(1u << (6 * i));
          const float ss = i < 2 ? sA.x : sB.x, zs = i < 2 ? sA.y : sB.y;
          const float sz = i < 2 ? zA.x : zB.x, zz = i < 2 ? zA.y : zB.y;
          kcs[i] = 8388608.f + zs * P;
          kms[i] = ss * (1.f / P);
          kcz[i] = 8388608.f + zz * P;
          kmz[i] = sz * (1.f / P);
        }
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const uint32_t q24 = f24[blk], z24 = f24[blk] >> 3;
          const float S0 = blk ? gB.x : gA.x, S1 = blk ? gB.y : gA.y;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t qb, zb2;
            if (i == 0) { qb = and_or<7u>(q24, kmagic); zb2 = and_or<7u>(z24, kmagic); }
            if (i == 1) { qb = and_or<7u << 6>(q24, kmagic); zb2 = and_or<7u << 6>(z24, kmagic); }
            if (i == 2) { qb = and_or<7u << 12>(q24, kmagic); zb2 = and_or<7u << 12>(z24, kmagic); }
            if (i == 3) { qb = and_or<7u << 18>(q24, kmagic); zb2 = and_or<7u << 18>(z24, kmagic); }
            const float sh = __fmul_rn(__fsub_rn(__uint_as_float(qb), kcs[i]), kms[i]);
            const float zh = __fmul_rn(__fsub_rn(__uint_as_float(zb2), kcz[i]), kmz[i]);
            const float C = blk ? c1[i] + e1[i] : c0[i] + e0[i];
            acc[i] = fmaf(sh, fmaf(-zh, (i & 1) ? S1 : S0, C), acc[i]);
          }
        }
      }
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
      if (++ls == (int)S) ls = 0;
    }
    // flush the row group: the lane's two columns, the outlier slots of rows g and g + 8 it
    // sums (lanes 8t .. 8t + 7), then the quad
    __syncwarp();
    float r0 = acc[0] + acc[1], r1 = acc[2] + acc[3];
    {
      float4* pa = reinterpret_cast<float4*>(myslots + g * 32 + 8 * t);
      float4* pb = reinterpret_cast<float4*>(myslots + (g + 8) * 32 + 8 * t);
      const float4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
      r0 += ((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w));
      r1 += ((b0.x + b0.y) + (b0.z + b0.w)) + ((b1.x + b1.y) + (b1.z + b1.w));
      const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
      pa[0] = z4;
      pa[1] = z4;
      pb[0] = z4;
      pb[1] = z4;
    }
    r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
    r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
    __syncwarp();
    if (t == 0) {
      fin.stage(cur_rg, rt * 16 + g, r0, done);
      fin.stage(cur_rg, rt * 16 + g + 8, r1, done);
    }
    ++cur_rg;
    kq = 0;
  }
  if (n_units == 0 && fin.rg0 >= 0 && t == 0) {  // an empty range inside a shared row group
    fin.stage(fin.rg0, rt * 16 + g, 0.f, done);
    fin.stage(fin.rg0, rt * 16 + g + 8, 0.f, done);
  }
  fin.finish(cs, threadIdx.x - grp * 128, done);
}

// ---------------------------------------------------------------------------------- W4

// ACT: act-order (v.perm set): the consumers gather x[perm] from the staged row; a separate
// instance, so that the static-group kernel carries none of that code
template <int STAGES, bool ACT>
__global__ void __launch_bounds__(kG1Threads, kG1CtasPerSm)
    w4_gemv1_kernel(W4View v, const uint16_t* __restrict__ X, uint16_t* __restrict__ Y, Workspace ws, G1Layout L) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* sb = smem_align128(smem_raw);
  G1Hdr& h = *reinterpret_cast<G1Hdr*>(sb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = v.G, U = (int64_t)v.RG * G, vN = v.N;
  float* gtab = reinterpret_cast<float*>(sb + L.gtab);
  uint16_t* xs = reinterpret_cast<uint16_t*>(sb + L.xs);
  uint32_t* xf = reinterpret_cast<uint32_t*>(sb + L.xf);
  const int g = lane >> 2, t = lane & 3;

  if (warp == 0) g1_plan_warp(h, U, G, lane, L);
  if (threadIdx.x == 32) {
#pragma unroll
    for (int q = 0; q < kG1Groups; ++q) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&h.full[q][s], 1);
        mbar_init(&h.empty[q][s], 128);  // every consumer thread of the group releases
      }
      mbar_init(&h.grp_bar[q], 128);
    }
    mbar_init(&h.all_bar, 32 * kG1Consumers);
    mbar_init(&h.x_bar, 1);
    mbar_init(&h.perm_bar, 1);
    fence_mbar_init();
    pdl_launch_dependents();
    if constexpr (ACT) {
      // act-order: the permutation entries of the K units this CTA stages (part of the
      // weights, so they go out now, with the plan's unit range computed here): read from
      // global memory by the gather itself they sat on the critical path of the CTAs that
      // start last (and took 32 registers)
      const int64_t W = (int64_t)gridDim.x * kG1Groups, c0 = (int64_t)blockIdx.x * kG1Groups;
      const int64_t a = g1_div(c0 * U, W, L.dW), n = g1_div((c0 + kG1Groups) * U, W, L.dW) - a;
      if (n > 0) {
        const int xn = (int)(n < G ? n : G);
        const int64_t ks = a - g1_div(a, G, L.dR) * G;
        const int na = (int)((int64_t)xn < G - ks ? (int64_t)xn : G - ks);
        int32_t* ps = reinterpret_cast<int32_t*>(sb + L.perm);
        mbar_arrive_expect_tx(&h.perm_bar, (uint32_t)xn * (kW4Group * 4));
        bulk_g2s(ps, v.perm + ks * kW4Group, (uint32_t)na * (kW4Group * 4), &h.perm_bar);
        if (xn > na) bulk_g2s(ps + (size_t)na * kW4Group, v.perm, (uint32_t)(xn - na) * (kW4Group * 4), &h.perm_bar);
      }
    }
  }
  __syncthreads();
  const int64_t u0c = h.u0[0], u1c = h.u0[kG1Groups];
  if (u1c <= u0c) return;

  if (warp >= kG1Consumers) {
    // ------------------------------------------- producers: one thread per group, own ring
    const int q = warp - kG1Consumers;
    if (q == 0 && lane == 1) {  // x, as soon as the previous kernel is done
      pdl_wait();  // x is written by the previous kernel on the stream
      if (ACT) {  // act-order: the whole row; the consumers gather from it
        mbar_arrive_expect_tx(&h.x_bar, (uint32_t)G * (kW4Group * 2));
        bulk_g2s(sb + L.xfull, X, (uint32_t)G * (kW4Group * 2), &h.x_bar);
      } else {
        const int xn = h.xn;
        const int64_t ks = u0c - g1_div(u0c, G, L.dR) * G;
        const int na = (int)((int64_t)xn < G - ks ? (int64_t)xn : G - ks);
        mbar_arrive_expect_tx(&h.x_bar, (uint32_t)xn * (kW4Group * 2));
        bulk_g2s(xs, X + ks * kW4Group, (uint32_t)na * (kW4Group * 2), &h.x_bar);
        if (xn > na) bulk_g2s(xs + (size_t)na * kW4Group, X, (uint32_t)(xn - na) * (kW4Group * 2), &h.x_bar);
      }
      return;
    }
    if (lane != 0) return;
    const int64_t a = h.u0[q];
    const int n = (int)(h.u0[q + 1] - a);
    const uint64_t pol = policy_evict_first();
    auto stage_at = [&](int s) { return sb + L.ring + (uint32_t)(q * STAGES + s) * L.stage_bytes; };
    auto unit_src = [&](int i) { return v.units + (a + i) * (int64_t)kW4UnitBytes; };
    const int pro = n < STAGES ? n : STAGES;
    int pf = pro + kG1W4Prefetch < n ? pro + kG1W4Prefetch : n;  // end of the prefetched window
    for (int i = 0; i < pro; ++i) {
      mbar_arrive_expect_tx(&h.full[q][i], kW4UnitBytes);
      bulk_g2s_ef(stage_at(i), unit_src(i), kW4UnitBytes, &h.full[q][i], pol);
    }
    if (pf > pro) prefetch_l2(unit_src(pro), (uint64_t)(pf - pro) * kW4UnitBytes);
    int s = 0;
    uint32_t ph = 1u;  // the ring's first pass is done: waiting for the consumers' first release
    for (int i = pro; i < n; ++i) {
      if (!g1_wait(&h.empty[q][s], ph ^ 1u, ws.status)) return;
      mbar_arrive_expect_tx(&h.full[q][s], kW4UnitBytes);
      bulk_g2s_ef(stage_at(s), unit_src(i), kW4UnitBytes, &h.full[q][s], pol);
      if (pf < n) {
        prefetch_l2(unit_src(pf), kW4UnitBytes);
        ++pf;
      }
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int grp = warp >> 2, rt = warp & 3;
  if constexpr (ACT) {
    // act-order: staged element j (K group (ks + j / 128) mod G, column j mod 128) is
    // x[perm[k]], gathered in shared memory from the whole row with the permutation entries
    // staged beside it
    const int nj = h.xn * kW4Group;
    pdl_wait();
    const bool got = g1_wait(&h.x_bar, 0, ws.status) && g1_wait(&h.perm_bar, 0, ws.status);
    const uint16_t* xrow = reinterpret_cast<const uint16_t*>(sb + L.xfull);
    const int32_t* ps = reinterpret_cast<const int32_t*>(sb + L.perm);
    if (got)
      for (int j = threadIdx.x; j < nj; j += 32 * kG1Consumers) xs[j] = xrow[ps[j]];
    named_bar_sync(1, 32 * kG1Consumers);  // every consumer thread, no early exit before it
    if (!got) return;
  } else {
    pdl_wait();
    if (!g1_wait(&h.x_bar, 0, ws.status)) return;
  }
  {
    // x in B-fragment order: per 128-group, lane column t, MMA j: the pairs (16j + 2t, +1)
    // and (16j + 2t + 8, +9), so that a lane reads its sixteen B registers of a group with
    // four 16-byte loads; every column of B carries the token
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(xs);
    const int nw = h.xn * 64;
    for (int i = threadIdx.x; i < nw; i += 32 * kG1Consumers) {
      const int lg = i >> 6, r = i & 63, tt = r >> 4, j = (r >> 1) & 7, hf = r & 1;
      xf[i] = xw[lg * 64 + 8 * j + tt + 4 * hf];
    }
    // sum of x per 128-group (one warp per group, fixed order)
    for (int lg = warp; lg < h.xn; lg += kG1Consumers) {
      const uint32_t p = xw[lg * 64 + lane], q = xw[lg * 64 + 32 + lane];
      float sum = (__uint_as_float(p << 16) + __uint_as_float(p & 0xFFFF0000u)) +
                  (__uint_as_float(q << 16) + __uint_as_float(q & 0xFFFF0000u));
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
      if (lane == 0) gtab[lg] = sum;
    }
  }
  mbar_arrive(&h.all_bar);
  if (!g1_wait(&h.all_bar, 0, ws.status)) return;

  const int64_t u0 = h.u0[grp];
  const int n_units = (int)(h.u0[grp + 1] - u0);
  const G1Fin fin{ws.tagged, h.own[grp], ws.status, ws.tag, (int)(blockIdx.x * kG1Groups + grp),
                  h.rg[grp][0], h.rg[grp][1], h.owned[grp], h.others[grp]};
  ConsumerSync cs{&h.grp_bar[grp], 0u, ws.status};
  auto done = [&](int64_t r, int row, float val) {
    const int64_t nrow = r * kRowGroup + row;
    if (nrow < vN) Y[nrow] = f2bf(val);
  };
  // this lane's offsets inside a stage and in the staged x
  const uint8_t* ring = sb + L.ring + (uint32_t)(grp * STAGES) * L.stage_bytes;
  const int code_off = ((rt * 2) * 32 + lane) * 16;           // k-block 1 at + 512
  const int stat_off = kW4CodeBytes + (rt * 16 + g) * 4;      // row g + 8 at + 32
  const uint32_t* xfl = xf + t * 16;                           // + 64 words per staged group
  const uint32_t kor = 0x43004300u;                            // bf16 128 + q

  int64_t cur_rg = h.rg0[grp];
  int kq = h.k0[grp], ls = h.ls0[grp], s = 0;
  uint32_t ph = 0;
  int it = 0;
  while (it < n_units) {
    // the units of one row group, then its flush
    const int seg_end = it + (int)G - kq < n_units ? it + (int)G - kq : n_units;
    float acc0 = 0.f, acc1 = 0.f;  // rows g and g + 8 of the tile (complete: every column is the token)
    for (; it < seg_end; ++it) {
      if (!g1_wait(&h.full[grp][s], ph, ws.status)) return;
      const uint8_t* unit = ring + s * L.stage_bytes;
      const uint32_t sz0 = *reinterpret_cast<const uint32_t*>(unit + stat_off);
      const uint32_t sz1 = *reinterpret_cast<const uint32_t*>(unit + stat_off + 32);
      const uint4 q0 = *reinterpret_cast<const uint4*>(unit + code_off);
      const uint4 q1 = *reinterpret_cast<const uint4*>(unit + code_off + 512);
      mbar_arrive(&h.empty[grp][s]);  // the stage's bytes are in registers
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
      const float Sg = gtab[ls];
      const uint4* xb = reinterpret_cast<const uint4*>(xfl + ls * 64);
      const uint4 xa = xb[0], xbb = xb[1], xc = xb[2], xd = xb[3];
      const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      const uint32_t bx[16] = {xa.x, xa.y, xa.z, xa.w, xbb.x, xbb.y, xbb.z, xbb.w,
                               xc.x, xc.y, xc.z, xc.w, xd.x, xd.y, xd.z, xd.w};
      // four independent accumulator chains over the eight k16 steps (two dependent MMAs each,
      // measured 2% faster than two chains of four); each starts from a zero C operand
      constexpr int NC = 4;
      float c[NC][4];
      const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w = words[j];
        uint32_t a[4];
        a[0] = and_or<0x000F000Fu>(w, kor);
        a[1] = and_or<0x000F000Fu>(w >> 4, kor);
        a[2] = and_or<0x000F000Fu>(w >> 8, kor);
        a[3] = and_or<0x000F000Fu>(w >> 12, kor);
        if (j < NC)
          mma_bf16_c(c[j % NC], a, bx[2 * j], bx[2 * j + 1], zero4);
        else
          mma_bf16(c[j % NC], a, bx[2 * j], bx[2 * j + 1]);
      }
      float r0 = c[0][0], r2 = c[0][2];
#pragma unroll
      for (int q = 1; q < NC; ++q) {
        r0 += c[q][0];
        r2 += c[q][2];
      }
      // sum (128 + q) x - (128 + z) sum x = sum (q - z) x, then the group's scale
      const float2 p0 = h2f2(sz0), p1 = h2f2(sz1);  // (scale, zero) of rows g and g + 8
      acc0 = fmaf(p0.x, fmaf(-(128.f + p0.y), Sg, r0), acc0);
      acc1 = fmaf(p1.x, fmaf(-(128.f + p1.y), Sg, r2), acc1);
      if (++ls == (int)G) ls = 0;
    }
    if (t == 0) {
      fin.stage(cur_rg, rt * 16 + g, acc0, done);
      fin.stage(cur_rg, rt * 16 + g + 8, acc1, done);
    }
    ++cur_rg;
    kq = 0;
  }
  if (n_units == 0 && fin.rg0 >= 0 && t == 0) {  // an empty range inside a shared row group
    fin.stage(fin.rg0, rt * 16 + g, 0.f, done);
    fin.stage(fin.rg0, rt * 16 + g + 8, 0.f, done);
  }
  fin.finish(cs, threadIdx.x - grp * 128, done);
}

// Layers below this many packed bytes get one CTA per SM instead of kG1CtasPerSm: the ring
// depth still leaves room for a second CTA, so the next forward's CTAs are all resident (and
// past their prologue) when this one ends, and for a small layer that start-up is a large
// part of the forward.  Measured, us per forward (one CTA per SM / two): W4 2048 x 4096
// 3.65 / 3.98, W4 4096^2 4.86 / 4.98 and act-order 5.41 / 6.72, SpQR 4096^2 5.58 / 6.00;
// above it W4 4096 x 5120 (11.1 MB) 5.54 / 5.09, SpQR 4096 x 6144 6.88 / 7.09 the other way.
constexpr int64_t kG1SmallBytes = 10ll << 20;
int g1_grid(int64_t U, int sms, bool spqr) {
  const int64_t bytes = U * (spqr ? kSpqrUnitBytes : kW4UnitBytes);
  const int64_t cps = bytes < kG1SmallBytes ? 1 : kG1CtasPerSm;
  int64_t grid = std::min<int64_t>(cps * sms, (U + kG1Groups - 1) / kG1Groups);
  if (spqr) grid = std::max<int64_t>(grid, (U + kG1MaxUnitsPerCta - 1) / kG1MaxUnitsPerCta);
  return (int)std::max<int64_t>(1, std::min<int64_t>(grid, 1 << 30));
}

// Launches with the deepest ring (of `deep` stages, or one less) whose shared memory fits.
template <typename KDeep, typename KShallow, typename View>
int g1_launch(KDeep* kdeep, KShallow* kshallow, int deep, std::atomic<uint64_t>* attr_done, const View& v, int64_t U,
              int64_t per_rg, bool spqr, bool xfull, const uint16_t* X, uint16_t* Y, const Workspace& ws,
              void* stream) {
  const int grid = g1_grid(U, ws.sms, spqr);
  if ((int64_t)grid * kG1Groups > ws.grid) return (int)cudaErrorInvalidValue;  // workspace slots
  const int xn = (int)std::min<int64_t>(per_rg, (U + grid - 1) / grid);
  const int xfull_k = xfull ? (int)(per_rg * kW4Group) : 0;
  // the deeper ring only if kG1CtasPerSm CTAs still share an SM: the grid assumes that many,
  // and one CTA fewer per SM runs the launch in two waves
  static std::atomic<int> sm_smem{0};
  if (sm_smem.load() == 0) {
    int dev = 0, per_sm = 0, reserved = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess)
      sm_smem.store(per_sm / kG1CtasPerSm - reserved);
    else
      cudaGetLastError();
  }
  const size_t share = sm_smem.load() > 0 ? (size_t)sm_smem.load() : kG1MaxSmem;
  int stages = deep;
  G1Layout L = g1_layout(spqr, xn, stages, xfull_k);
  if ((size_t)L.bytes + 128 > std::min(share, kG1MaxSmem)) {
    stages = deep - 1;
    L = g1_layout(spqr, xn, stages, xfull_k);
  }
  if (U >= (int64_t(1) << 32) || per_rg >= (int64_t(1) << 32)) return (int)cudaErrorInvalidValue;
  L.dW = g1_div_make((uint32_t)grid * kG1Groups);
  L.dU = g1_div_make((uint32_t)U);
  L.dR = g1_div_make((uint32_t)per_rg);
  const size_t smem = (size_t)L.bytes + 128;
  if (smem > kG1MaxSmem) return (int)cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kG1Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = QLIN_USE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the shared-memory limit is raised once per device to the largest size any layer needs
  if (stages == deep) {
    if (const int e = smem_attr_once(kdeep, kG1MaxSmem, attr_done[0])) return e;
    return (int)cudaLaunchKernelEx(&cfg, kdeep, v, X, Y, ws, L);
  }
  if (const int e = smem_attr_once(kshallow, kG1MaxSmem, attr_done[1])) return e;
  return (int)cudaLaunchKernelEx(&cfg, kshallow, v, X, Y, ws, L);
}

}  // namespace

int gemv1_slots(int64_t units, int sms, bool spqr) { return g1_grid(units, sms, spqr) * kG1Groups; }

int launch_spqr_gemv1(const SpqrView& v, const uint16_t* X, uint16_t* Y, const Workspace& ws, void* stream) {
  static std::atomic<uint64_t> attr_done[2];
  return g1_launch(spqr_gemv1_kernel<kG1SpStages>, spqr_gemv1_kernel<kG1SpStages - 1>, kG1SpStages, attr_done, v,
                   (int64_t)v.RG * v.S, v.S, true, false, X, Y, ws, stream);
}

int launch_w4_gemv1(const W4View& v, const uint16_t* X, uint16_t* Y, const Workspace& ws, void* stream) {
  static std::atomic<uint64_t> attr_done[4];
  if (v.perm)
    return g1_launch(w4_gemv1_kernel<kG1W4Stages, true>, w4_gemv1_kernel<kG1W4Stages - 1, true>, kG1W4Stages,
                     attr_done + 2, v, (int64_t)v.RG * v.G, v.G, false, true, X, Y, ws, stream);
  return g1_launch(w4_gemv1_kernel<kG1W4Stages, false>, w4_gemv1_kernel<kG1W4Stages - 1, false>, kG1W4Stages,
                   attr_done, v, (int64_t)v.RG * v.G, v.G, false, false, X, Y, ws, stream);
}

}  // namespace qlin

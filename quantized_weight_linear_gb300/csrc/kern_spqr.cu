// SpQR decode GEMV for 2 <= M <= 16 tokens: Y = X (D + S)^T, dense 3-bit bi-level part D
// and fp16 outliers S applied in the same pass.  (One token: kern_gemv1.cu.)
//
// SpQR page ("Makale Bülteni — SpQR", "İddia ve Gerçeklik: SpQR"): the kernel unpacks the
// dense 3-bit codes while it runs the sparse fp16 product, and the page warns that
// register pressure and warp divergence are the cost of the hybrid.  Design here:
//
// * a persistent weight stream: up to three CTAs per SM, equal contiguous ranges of
//   (64 rows x 256-wide supergroup) units (7424 bytes of codes, 3-bit group statistics and
//   fp16 supergroup statistics), a producer warp with cp.async.bulk into a 2-deep ring per
//   CTA, the unit's outlier bucket and X slice staged alongside (the slice is two 2D tensor
//   copies of all M rows, not one copy per token);
// * code words hold five 3-bit fields per 16-bit half; one AND/OR turns a field pair into
//   bf16 (base + q) with base 128 or 16 depending on the field;
// * the A pairs are dequantized to bf16 s^ (q - z^) in registers and the MMA columns carry
//   the tokens;
// * outliers: each warp keeps a shared-memory table with one bf16 slot per (MMA step, lane, A
//   register, half), seeded with the register's -s^ z^; its row tile's bucket (k < 256,
//   row < 16, fp16 value) is added into the slots, and every MMA step takes its row of the
//   table as the addend of the FMA that dequantizes its A registers.  An outlier then costs
//   the same at any token count, no two lanes ever write one slot (no atomics), and the steps
//   carry no branch (the page's warning about the sparse part is about exactly this
//   scattered accumulation and its divergence).
#include "kern_decode_common.cuh"

namespace qlin {
namespace {

#ifndef QLIN_SP_DEC_STAGES
#define QLIN_SP_DEC_STAGES 2  // two: room for the outlier-correction table at three CTAs per SM
#endif
constexpr int kStagesSp = QLIN_SP_DEC_STAGES;
constexpr int kXHalfSp = 136;      // each 128-wide half of the X slice as [XR][128 + 8 pad]
constexpr int kOutCap = 640;       // outlier entries staged per unit (more -> read from global)
constexpr int kOffsCap = 1024 + 16;  // offsets staged per CTA

template <int XR>  // staged X rows (8 or 16)
struct SpSmem {
  static constexpr int kXE = 2 * XR * kXHalfSp;  // X elements per stage
  __align__(128) uint8_t unit[kStagesSp][kSpqrUnitBytes];
  __align__(128) uint16_t x[kStagesSp][kXE];
  __align__(16) uint32_t out[kStagesSp][kOutCap + 8];
  __align__(16) uint32_t offs[kOffsCap];
  float own[kRowGroup * 4];  // M <= 4: this CTA's partial sums of the row group it owns
  // per consumer warp, MMA step and lane, the bf16 additive terms of the lane's A registers
  // (-s^ z^ of the register's (row, group), plus the outlier where the weight has one), all 16
  // steps of a unit; a step's row of 32 lanes is contiguous, so its loads are free of bank
  // conflicts
  __align__(16) uint32_t otab[4][16][32][4];
  uint64_t full[kStagesSp];
  uint64_t empty[kStagesSp];
  uint64_t offs_bar;
  uint64_t cons_bar;
  int flags[2];
};

// bucket bounds of unit u, row tile rt, from the staged offsets
struct OffsView {
  const uint32_t* s;
  int64_t base;  // global index of s[0]
  __device__ __forceinline__ uint32_t operator()(int64_t i) const { return s[i - base]; }
};

// A register pair for MMA j, register r, from the lane's six code words (bf16 base + q).
template <int J, int R>
__device__ __forceinline__ uint32_t spqr_pair(const uint32_t (&w)[6]) {
  if constexpr (J <= 4) {
    constexpr int i = 4 * J + R;
    if constexpr (i < 18) {
      constexpr int wi = i / 3, f = (i % 3) * 2;
      return lop_and_or(w[wi] >> (3 * f), 0x00070007u, 0x43004300u);
    } else {
      constexpr int b = 3 * (i - 18);
      return ((w[b] >> 15) & 0x00010001u) | ((w[b + 1] >> 14) & 0x00020002u) |
             ((w[b + 2] >> 13) & 0x00040004u) | 0x43004300u;
    }
  } else {
    constexpr int i = 4 * (J - 5) + R;
    constexpr int wi = i / 2, f = (i % 2) * 2 + 1;
    return lop_and_or(w[wi] >> (3 * (f - 1)), 0x00380038u, 0x41804180u);
  }
}

template <int J>
__device__ __forceinline__ void spqr_frag(const uint32_t (&w)[6], uint32_t (&a)[4]) {
  a[0] = spqr_pair<J, 0>(w);
  a[1] = spqr_pair<J, 1>(w);
  a[2] = spqr_pair<J, 2>(w);
  a[3] = spqr_pair<J, 3>(w);
}

// 6-bit (qs, qz) entry of (row r_in_tile, group gb in block) from the block's 96-byte field area
__device__ __forceinline__ uint32_t qsqz_entry(const uint8_t* area, int r, int gb) {
  const int lane = 4 * (r & 7) + (gb >> 1);
  const int i = ((r >> 3) << 1) | (gb & 1);
  const int bit = 24 * lane + 6 * i;
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(area);
  const uint32_t lo = wp[bit >> 5], hi = wp[(bit >> 5) + 1];
  return __funnelshift_r(lo, hi, bit & 31) & 63u;
}

#ifndef QLIN_SP_CPS16
#define QLIN_SP_CPS16 3
#endif
template <int MT, int OWN>  // MT: 8-token column tiles (M <= 8 MT); OWN: see below
__global__ void __launch_bounds__(160, MT == 1 ? 3 : QLIN_SP_CPS16)
    spqr_decode_kernel(const __grid_constant__ CUtensorMap xmap, SpqrView v, const uint16_t* __restrict__ X,
                       uint16_t* __restrict__ Y, int M, Workspace ws) {
  constexpr int XR = 8 * MT;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SpSmem<XR>& sm = *reinterpret_cast<SpSmem<XR>*>(smem_align128(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t grid = gridDim.x, cta = blockIdx.x;
  // scalars of the view as locals: lambdas capture them, and capturing the kernel parameter
  // itself would move it to local memory
  const int64_t vN = v.N;
  const int64_t S = v.S, U = (int64_t)v.RG * S;
  const int64_t u0 = split_start(cta, U, grid), u1 = split_start(cta + 1, U, grid);
  const int n_units = (int)(u1 - u0);
  // staged offsets: global indices [4 u0, 4 u1] (aligned down to 16 bytes)
  const int64_t off_base = (u0 * 4) & ~int64_t(3);
  const int64_t off_end = (u1 * 4 + 1 + 3) & ~int64_t(3);
  const OffsView offs{sm.offs, off_base};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesSp; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 4);
    }
    mbar_init(&sm.offs_bar, 1);
    mbar_init(&sm.cons_bar, 128);
    fence_mbar_init();
    pdl_launch_dependents();
  }
  {
    uint32_t* xz = reinterpret_cast<uint32_t*>(&sm.x[0][0]);
    for (int i = threadIdx.x; i < kStagesSp * SpSmem<XR>::kXE / 2; i += blockDim.x) xz[i] = 0u;
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == 4) {
    if (lane != 0) return;
    mbar_arrive_expect_tx(&sm.offs_bar, (uint32_t)(off_end - off_base) * 4);
    bulk_g2s(sm.offs, v.offs + off_base, (uint32_t)(off_end - off_base) * 4, &sm.offs_bar);
    if (!mbar_wait(&sm.offs_bar, 0, ws.status)) return;
    auto weights = [&](int s, int64_t u) -> uint32_t {  // returns bytes issued
      bulk_g2s(sm.unit[s], v.units + u * (int64_t)kSpqrUnitBytes, kSpqrUnitBytes, &sm.full[s]);
      const uint32_t e0 = offs(4 * u), e1 = offs(4 * u + 4);
      uint32_t bytes = kSpqrUnitBytes;
      if (e1 - e0 <= (uint32_t)kOutCap && e1 > e0) {
        const uint32_t a0 = e0 & ~3u, a1 = (e1 + 3u) & ~3u;
        bulk_g2s(sm.out[s], v.ents + a0, (a1 - a0) * 4, &sm.full[s]);
        bytes += (a1 - a0) * 4;
      }
      return bytes;
    };
    auto out_bytes = [&](int64_t u) -> uint32_t {
      const uint32_t e0 = offs(4 * u), e1 = offs(4 * u + 4);
      if (e1 - e0 <= (uint32_t)kOutCap && e1 > e0) return (((e1 + 3u) & ~3u) - (e0 & ~3u)) * 4;
      return 0u;
    };
    // M == 1: one plain copy of the 256-wide slice; otherwise two boxes of xmap ([M][136] at
    // k0 and k0 + 128), one per half of the staged layout
    const uint32_t xtx = 2u * (uint32_t)M * kXHalfSp * 2;
    int kx = (int)(u0 % S);  // supergroup of the next X slice (units are issued in order)
    auto load_x = [&](int s) {
      const int k0 = kx * kSpqrSuper;
      if (++kx == (int)S) kx = 0;
      tma_load_2d(&sm.x[s][0], &xmap, k0, 0, &sm.full[s]);
      tma_load_2d(&sm.x[s][XR * kXHalfSp], &xmap, k0 + 128, 0, &sm.full[s]);
    
    };
    const int pro = n_units < kStagesSp ? n_units : kStagesSp;
    for (int i = 0; i < pro; ++i) {
      mbar_arrive_expect_tx(&sm.full[i], kSpqrUnitBytes + out_bytes(u0 + i) + xtx);
      weights(i, u0 + i);
    }
    pdl_wait();
    for (int i = 0; i < pro; ++i) load_x(i);
    for (int i = kStagesSp; i < n_units; ++i) {
      const int s = i % kStagesSp;
      const uint32_t ph = (uint32_t)(i / kStagesSp) & 1u;
      if (!mbar_wait(&sm.empty[s], ph ^ 1u, ws.status)) return;
      mbar_arrive_expect_tx(&sm.full[s], kSpqrUnitBytes + out_bytes(u0 + i) + xtx);
      weights(s, u0 + i);
      load_x(s);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  const int rt = warp;
  ConsumerSync cs{&sm.cons_bar, 0u, ws.status};
  if (!mbar_wait(&sm.offs_bar, 0, ws.status)) return;
  constexpr int NACC = 4 * MT;
  float acc[NACC];
#pragma unroll
  for (int i = 0; i < NACC; ++i) acc[i] = 0.f;
  int64_t cur_rg = u0 / S;
  UnitCursor cur{cur_rg, (int)(u0 - cur_rg * S), (int)S};

  constexpr int NV = NACC;
  int idx[NV];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = g + ((i & 2) ? 8 : 0);
      const int m = 2 * t + (i & 1) + 8 * mt;
      idx[mt * 4 + i] = (m < M) ? (rt * 16 + r) * 16 + m : -1;
    }
  auto done = [&](int64_t rg, const float (&out)[NV]) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (idx[j] < 0) continue;
      const int64_t n = rg * kRowGroup + idx[j] / 16;
      const int m = idx[j] % 16;
      if (n < vN) Y[(int64_t)m * vN + n] = f2bf(out[j]);
    }
  };
  // up to OWN (1 or 4) tokens: the owner-reduces completion (no atomics); otherwise counted
  auto fin = [&] {
    if constexpr (OWN > 0)
      return OwnerFinisher<NV, OWN>(S, U, grid, cta, ws.tagged, ws.tag, ws.status, sm.own);
    else
      return RowGroupFinisher<float, NV>(S, U, grid, cta, ws.partials, ws.counters);
  }();
  auto flush = [&](int64_t rg) { fin.stage(rg, acc, idx, done); };

  // the previous kernel on the stream may still read this launch's outputs or workspace
  pdl_wait();
  for (int it = 0; it < n_units; ++it) {
    const int s = it % kStagesSp;
    const uint32_t ph = (uint32_t)(it / kStagesSp) & 1u;
    const int64_t u = u0 + it;
    const int64_t rg = cur.rg;
    cur.next();
    if (rg != cur_rg) {
      flush(cur_rg);
#pragma unroll
      for (int i = 0; i < NACC; ++i) acc[i] = 0.f;
      cur_rg = rg;
    }
    if (!mbar_wait(&sm.full[s], ph, ws.status)) return;
    const uint8_t* unit = sm.unit[s];
    const uint16_t* sgst = reinterpret_cast<const uint16_t*>(unit + kSpqrCodeBytes + kSpqrQsqzBytes);
    const uint16_t* ra = sgst + (rt * 16 + g) * 4;
    const uint16_t* rb = sgst + (rt * 16 + g + 8) * 4;
    const float ssA = h2f_dev(ra[0]), zsA = h2f_dev(ra[1]), szA = h2f_dev(ra[2]), zzA = h2f_dev(ra[3]);
    const float ssB = h2f_dev(rb[0]), zsB = h2f_dev(rb[1]), szB = h2f_dev(rb[2]), zzB = h2f_dev(rb[3]);
    // the unit's four bucket starts in one 16-byte load (the staged offsets start at 4 u0)
    const uint4 o4 = *reinterpret_cast<const uint4*>(&sm.offs[4 * it]);
    const uint32_t e0 = o4.x, e1 = offs(4 * u + 4);
    const uint32_t b0 = rt == 0 ? o4.x : rt == 1 ? o4.y : rt == 2 ? o4.z : o4.w;
    const uint32_t b1 = rt == 0 ? o4.y : rt == 1 ? o4.z : rt == 2 ? o4.w : e1;
    const bool staged = (e1 - e0 <= (uint32_t)kOutCap) && e1 > e0;
    const uint32_t* bs = sm.out[s] + (b0 - (e0 & ~3u));  // staged bucket
    const uint32_t* bg = v.ents + b0;               // the same bucket in global memory
    const int n = (int)(b1 - b0);

    // A-side statistics of both blocks: (row g, group t), (row g+8, group t), (row g, group
    // t+4), (row g+8, group t+4)
    uint32_t sh2[2][4], ch2[2][4];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint8_t* qarea = unit + kSpqrCodeBytes + (rt * 2 + blk) * 96;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = g + ((r & 1) ? 8 : 0), gb = t + ((r & 2) ? 4 : 0);
        const uint32_t e = qsqz_entry(qarea, row, gb);
        const float ss = (r & 1) ? ssB : ssA, zs = (r & 1) ? zsB : zsA;
        const float sz = (r & 1) ? szB : szA, zz = (r & 1) ? zzB : zzA;
        const float sh = __fmul_rn(__fsub_rn((float)(e & 7u), zs), ss);
        const float zh = __fmul_rn(__fsub_rn((float)(e >> 3), zz), sz);
        sh2[blk][r] = pack_bf16x2(sh, sh);
        const float cz = -sh * zh;
        ch2[blk][r] = pack_bf16x2(cz, cz);
      }
    }
    // The table: every slot of this lane starts at its register's -s^ z^, and the outliers are
    // added into it, so each MMA step dequantizes its A registers with one bf16x2 FMA whose
    // addend is the table row: bf16((q - base) s^ + t), t = -s^ z^ or bf16(-s^ z^ + s).  Entry
    // i of the (unit, row tile) bucket goes to the slot of the lane and register that hold
    // its weight (element 2j + (k & 1) of group G = (k & 127) / 16: lane 4 (row & 7) + (G & 3),
    // register (row >> 3) + 2 (G >> 2), step 8 (k / 128) + j); every position is unique, so
    // the 16-bit read-modify-writes never collide.  (A walk per row and token took a third of
    // the kernel; a branch in the unrolled steps broke their scheduling; at sixteen tokens a
    // table of one 128-wide block, filled before each block, was 6% slower on 70B-class
    // layers.)  The fill also overwrites whatever the previous unit left in the lane's slots.
#pragma unroll
    for (int q = 0; q < 16; ++q)
      *reinterpret_cast<uint4*>(sm.otab[rt][q][lane]) =
          make_uint4(ch2[q >> 3][0], ch2[q >> 3][1], ch2[q >> 3][2], ch2[q >> 3][3]);
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      uint32_t e;
      if (staged)
        e = bs[i];
      else
        e = __ldg(bg + i);
      const int kin = (int)((e >> 4) & 255u);
      const int row = (int)(e & 15u), kb = kin & 127;
      uint16_t* p = reinterpret_cast<uint16_t*>(
          &sm.otab[rt][(kin >> 7) * 8 + ((kb & 15) >> 1)][4 * (row & 7) + ((kb >> 4) & 3)][(row >> 3) | ((kb >> 6) << 1)]);
      p[kin & 1] = f2bf(bf2f(p[kin & 1]) + h2f_dev((uint16_t)(e >> 16)));
    }
    __syncwarp();
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t* cw = reinterpret_cast<const uint32_t*>(unit) + ((rt * 2 + blk) * 32 + lane) * 6;
      uint32_t w[6];
      {
        const uint2 p0 = *reinterpret_cast<const uint2*>(cw);
        const uint2 p1 = *reinterpret_cast<const uint2*>(cw + 2);
        const uint2 p2 = *reinterpret_cast<const uint2*>(cw + 4);
        w[0] = p0.x; w[1] = p0.y; w[2] = p1.x; w[3] = p1.y; w[4] = p2.x; w[5] = p2.y;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t a[4];
        switch (j) {
          case 0: spqr_frag<0>(w, a); break;
          case 1: spqr_frag<1>(w, a); break;
          case 2: spqr_frag<2>(w, a); break;
          case 3: spqr_frag<3>(w, a); break;
          case 4: spqr_frag<4>(w, a); break;
          case 5: spqr_frag<5>(w, a); break;
          case 6: spqr_frag<6>(w, a); break;
          default: spqr_frag<7>(w, a); break;
        }
        const uint32_t base = j <= 4 ? 0x43004300u : 0x41804180u;
        {
          const uint4 d = *reinterpret_cast<const uint4*>(sm.otab[rt][8 * blk + j][lane]);
          a[0] = bf16x2_fma(bf16x2_sub(a[0], base), sh2[blk][0], d.x);
          a[1] = bf16x2_fma(bf16x2_sub(a[1], base), sh2[blk][1], d.y);
          a[2] = bf16x2_fma(bf16x2_sub(a[2], base), sh2[blk][2], d.z);
          a[3] = bf16x2_fma(bf16x2_sub(a[3], base), sh2[blk][3], d.w);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint16_t* xr = &sm.x[s][(blk * XR + g + 8 * mt) * kXHalfSp];
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xr + 16 * t + 2 * j);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(xr + 16 * (t + 4) + 2 * j);
          mma_bf16_4(acc[mt * 4 + 0], acc[mt * 4 + 1], acc[mt * 4 + 2], acc[mt * 4 + 3], a, b0, b1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
  }
  if (n_units > 0) {
    flush(cur_rg);
    fin.finish(M, cs, sm.flags, [&](int64_t rg, int e, float val) {
      const int64_t n = rg * kRowGroup + e / 16;
      if (n < vN) Y[(int64_t)(e % 16) * vN + n] = f2bf(val);
    });
  }
}

static_assert(offsetof(SpSmem<8>, x) % 128 == 0 && offsetof(SpSmem<16>, x) % 128 == 0 &&
                  (SpSmem<8>::kXE * 2) % 128 == 0 && (SpSmem<16>::kXE * 2) % 128 == 0 && (8 * kXHalfSp * 2) % 128 == 0,
              "TMA destinations");

template <int MT, int OWN>
int launch_spqr_t(const SpqrView& v, const uint16_t* X, uint16_t* Y, int M, const Workspace& ws, int grid,
                  void* stream) {
  constexpr int XR = 8 * MT;
  CUtensorMap xmap{};
  if (!encode_decode_x_map(&xmap, X, v.K, M, kXHalfSp)) return (int)cudaErrorInvalidValue;
  const size_t smem = sizeof(SpSmem<XR>) + 128;
  static std::atomic<uint64_t> attr_done{0};
  if (const int e = smem_attr_once(spqr_decode_kernel<MT, OWN>, smem, attr_done)) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(160);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = QLIN_USE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, spqr_decode_kernel<MT, OWN>, xmap, v, X, Y, M, ws);
}

}  // namespace

int spqr_decode_grid(const SpqrView& v, int M, int sms) {
  // several CTAs per SM hide the unpack latency; every CTA stages its slice of the bucket
  // offsets, so ranges stay below kOffsCap entries
  const int64_t U = (int64_t)v.RG * v.S;
  const int cps = std::min(M <= 8 ? 3 : QLIN_SP_CPS16, QLIN_DECODE_CPS_MAX);
  int64_t grid = std::min<int64_t>(U, (int64_t)cps * sms);
  const int64_t need = (U * 4 + (kOffsCap - 24) - 1) / (kOffsCap - 24);
  if (grid < need) grid = std::min<int64_t>(U, need);
  return (int)std::min<int64_t>(grid, 1 << 30);
}

int launch_spqr_decode(const SpqrView& v, const uint16_t* X, uint16_t* Y, int M, const Workspace& ws, int grid,
                       void* stream) {
  if (M == 1) return launch_spqr_gemv1(v, X, Y, ws, stream);
  grid = spqr_decode_grid(v, M, ws.sms);
  if (grid > ws.grid) return (int)cudaErrorInvalidValue;
  if (M <= 4) return launch_spqr_t<1, 4>(v, X, Y, M, ws, grid, stream);
  if (M <= 8) return launch_spqr_t<1, 0>(v, X, Y, M, ws, grid, stream);
  return launch_spqr_t<2, 0>(v, X, Y, M, ws, grid, stream);
}

}  // namespace qlin

// W4 g128 decode GEMV for 2 <= M <= 16 tokens: Y[m, n] = sum_k x[m, k] * (q[n, k] - z) * s.
// (One token: kern_gemv1.cu.)
//
// GPTQ page ("Makale Bülteni — GPTQ", "İddia ve Gerçeklik: GPTQ"): weight-only 4-bit
// groups pay off at small batch because the layer is bound by weight bandwidth.  The
// kernel is therefore a weight stream:
//
// * persistent grid of up to four CTAs per SM, each owning an equal, contiguous range of
//   (64-row group, 128-wide K group) units (4352 bytes of codes + statistics each);
// * one producer warp streams units with cp.async.bulk into a 4-deep shared-memory
//   ring (mbarrier full/empty pairs) together with the matching 128-wide slice of X (with
//   two or more tokens one 2D tensor copy of all M rows, not one copy per token);
// * four consumer warps (one 16-row tile each) turn code words into bf16 A fragments
//   with one AND/OR per register pair (bf16 128 + q) and one bf16 subtract of 128 + z,
//   which leaves the exact integers q - z; mma.sync m16n8k16 accumulates sum (q - z) x in
//   fp32 per group, and the group's fp16 scale is applied once per group;
// * a row group split between CTAs is finished deterministically: with up to four tokens by
//   the CTA that owns it (tagged partial words, no atomics), otherwise by the last CTA to
//   arrive (partials in the workspace, arrival counter).
#include "kern_decode_common.cuh"

namespace qlin {
namespace {

constexpr int kStagesW4 = 4;
constexpr int kXStrideW4 = 136;  // staged X row: 128 bf16 + 8 pad (bank-conflict free B loads)

template <int MT>
struct W4Smem {
  __align__(128) uint8_t unit[kStagesW4][kW4UnitBytes];
  __align__(128) uint16_t x[kStagesW4][8 * MT][kXStrideW4];  // stage stride 2176 * MT bytes
  uint64_t full[kStagesW4];
  uint64_t empty[kStagesW4];
  uint64_t cons_bar;
  int flags[2];
  float own[kRowGroup * 4];  // up to 4 tokens: this CTA's partial sums of the row group it owns
};

#ifndef QLIN_W4_CPS16
#define QLIN_W4_CPS16 3
#endif
template <int MT, int OWN>  // OWN: 4 (M <= 4, owner-reduces split completion), 0 counted
__global__ void __launch_bounds__(160, MT == 1 ? 4 : QLIN_W4_CPS16)
    w4_decode_kernel(const __grid_constant__ CUtensorMap xmap, W4View v, const uint16_t* __restrict__ X,
                     uint16_t* __restrict__ Y, int M, Workspace ws) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  W4Smem<MT>& sm = *reinterpret_cast<W4Smem<MT>*>(smem_align128(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t grid = gridDim.x, cta = blockIdx.x;
  // scalars of the view as locals: lambdas capture them, and capturing the kernel parameter
  // itself would move it to local memory
  const int64_t vN = v.N;
  const int64_t G = v.G, U = (int64_t)v.RG * G;
  const int64_t u0 = split_start(cta, U, grid), u1 = split_start(cta + 1, U, grid);
  const int n_units = (int)(u1 - u0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesW4; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 4);
    }
    mbar_init(&sm.cons_bar, 128);
    fence_mbar_init();
    pdl_launch_dependents();
  }
  {
    uint32_t* xz = reinterpret_cast<uint32_t*>(&sm.x[0][0][0]);
    for (int i = threadIdx.x; i < kStagesW4 * 8 * MT * kXStrideW4 / 2; i += blockDim.x) xz[i] = 0u;
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == 4) {
    if (lane != 0) return;
    const uint32_t xbytes = (uint32_t)M * kXStrideW4 * 2;  // one box of xmap: [M][136] at k0
    const uint32_t tx = kW4UnitBytes + xbytes;
    int kx = (int)(u0 % G);  // K group of the next X slice (units are issued in order)
    auto load_x = [&](int s) {
      const int k0 = kx * kW4Group;
      tma_load_2d(&sm.x[s][0][0], &xmap, k0, 0, &sm.full[s]);
      if (++kx == (int)G) kx = 0;
    };
    const int pro = n_units < kStagesW4 ? n_units : kStagesW4;
    for (int i = 0; i < pro; ++i) {
      mbar_arrive_expect_tx(&sm.full[i], tx);
      bulk_g2s(sm.unit[i], v.units + (u0 + i) * (int64_t)kW4UnitBytes, kW4UnitBytes, &sm.full[i]);
    }
    pdl_wait();  // X is written by the previous kernel on the stream
    for (int i = 0; i < pro; ++i) load_x(i);
    for (int i = kStagesW4; i < n_units; ++i) {
      const int s = i % kStagesW4;
      const uint32_t ph = (uint32_t)(i / kStagesW4) & 1u;
      if (!mbar_wait(&sm.empty[s], ph ^ 1u, ws.status)) return;
      mbar_arrive_expect_tx(&sm.full[s], tx);
      bulk_g2s(sm.unit[s], v.units + (u0 + i) * (int64_t)kW4UnitBytes, kW4UnitBytes, &sm.full[s]);
      load_x(s);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  ConsumerSync cs{&sm.cons_bar, 0u, ws.status};
  float acc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;
  int64_t cur_rg = u0 / G;
  UnitCursor cur{cur_rg, (int)(u0 - cur_rg * G), (int)G};

  int idx[MT * 4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = warp * 16 + g + ((i & 2) ? 8 : 0);
      const int m = 2 * t + (i & 1) + 8 * mt;
      idx[mt * 4 + i] = (m < M) ? r * 16 + m : -1;
    }
  auto done = [&](int64_t rg, const float (&out)[MT * 4]) {
#pragma unroll
    for (int j = 0; j < MT * 4; ++j) {
      if (idx[j] < 0) continue;
      const int64_t n = rg * kRowGroup + idx[j] / 16;
      const int m = idx[j] % 16;
      if (n < vN) Y[(int64_t)m * vN + n] = f2bf(out[j]);
    }
  };
  auto fin = [&] {
    if constexpr (OWN > 0)
      return OwnerFinisher<MT * 4, OWN>(G, U, grid, cta, ws.tagged, ws.tag, ws.status, sm.own);
    else
      return RowGroupFinisher<float, MT * 4, MT == 1 ? 16 : 8>(G, U, grid, cta, ws.partials, ws.counters);
  }();
  auto flush = [&](int64_t rg) {
    float vals[MT * 4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) vals[mt * 4 + i] = acc[mt][i];
    fin.stage(rg, vals, idx, done);
  };

  // the previous kernel on the stream may still read this launch's outputs or workspace
  pdl_wait();
  for (int i = 0; i < n_units; ++i) {
    const int s = i % kStagesW4;
    const uint32_t ph = (uint32_t)(i / kStagesW4) & 1u;
    const int64_t rg = cur.rg;
    cur.next();
    if (rg != cur_rg) {
      flush(cur_rg);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[mt][q] = 0.f;
      cur_rg = rg;
    }
    if (!mbar_wait(&sm.full[s], ph, ws.status)) return;
    const uint8_t* unit = sm.unit[s];
    const uint32_t* st = reinterpret_cast<const uint32_t*>(unit + kW4CodeBytes);
    const uint32_t sz0 = st[warp * 16 + g], sz1 = st[warp * 16 + g + 8];
    const float s0 = h2f_dev((uint16_t)(sz0 & 0xFFFFu)), s1 = h2f_dev((uint16_t)(sz1 & 0xFFFFu));
    const float z0 = h2f_dev((uint16_t)(sz0 >> 16)), z1 = h2f_dev((uint16_t)(sz1 >> 16));
    const uint32_t zp0 = pack_bf16x2(128.f + z0, 128.f + z0);
    const uint32_t zp1 = pack_bf16x2(128.f + z1, 128.f + z1);
    // two accumulator chains per tile (even / odd k16 step) keep the MMA pipe busy
    float c[2 * MT][4];
#pragma unroll
    for (int mt = 0; mt < 2 * MT; ++mt)
#pragma unroll
      for (int q = 0; q < 4; ++q) c[mt][q] = 0.f;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      const uint4 wv = *reinterpret_cast<const uint4*>(unit + ((warp * 2 + kb) * 32 + lane) * 16);
      const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = words[j];
        uint32_t a[4];
        a[0] = bf16x2_sub(lop_and_or(w, 0x000F000Fu, 0x43004300u), zp0);
        a[1] = bf16x2_sub(lop_and_or(w >> 4, 0x000F000Fu, 0x43004300u), zp1);
        a[2] = bf16x2_sub(lop_and_or(w >> 8, 0x000F000Fu, 0x43004300u), zp0);
        a[3] = bf16x2_sub(lop_and_or(w >> 12, 0x000F000Fu, 0x43004300u), zp1);
        const int kk = kb * 64 + 16 * j + 2 * t;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint16_t* xr = &sm.x[s][g + 8 * mt][0];
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xr + kk);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(xr + kk + 8);
          mma_bf16(c[2 * mt + (j & 1)], a, b0, b1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      acc[mt][0] += s0 * (c[2 * mt][0] + c[2 * mt + 1][0]);
      acc[mt][1] += s0 * (c[2 * mt][1] + c[2 * mt + 1][1]);
      acc[mt][2] += s1 * (c[2 * mt][2] + c[2 * mt + 1][2]);
      acc[mt][3] += s1 * (c[2 * mt][3] + c[2 * mt + 1][3]);
    }
  }
  if (n_units > 0) {
    flush(cur_rg);
    fin.finish(M, cs, sm.flags, [&](int64_t rg, int e, float val) {
      const int64_t n = rg * kRowGroup + e / 16;
      if (n < vN) Y[(int64_t)(e % 16) * vN + n] = f2bf(val);
    });
  }
}

static_assert(offsetof(W4Smem<1>, x) % 128 == 0 && offsetof(W4Smem<2>, x) % 128 == 0, "TMA destination");

template <int MT, int OWN>
int launch_w4_mt(const W4View& v, const uint16_t* X, uint16_t* Y, int M, const Workspace& ws, int grid,
                 void* stream) {
  CUtensorMap xmap{};
  if (!encode_decode_x_map(&xmap, X, v.K, M, kXStrideW4)) return (int)cudaErrorInvalidValue;
  const size_t smem = sizeof(W4Smem<MT>) + 128;
  static std::atomic<uint64_t> attr_done{0};
  if (const int e = smem_attr_once(w4_decode_kernel<MT, OWN>, smem, attr_done)) return e;
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
  return (int)cudaLaunchKernelEx(&cfg, w4_decode_kernel<MT, OWN>, xmap, v, X, Y, M, ws);
}

}  // namespace

namespace {

// Act-order layers (GPTQ page, "İddia ve Gerçeklik: GPTQ", last paragraph): the codes are in
// the permuted column order, so the activations are gathered into it first,
// Xp[m][j] = X[m][perm[j]], eight channels per thread and one 16-byte store.
__global__ void __launch_bounds__(256)
    w4_gather_kernel(const uint16_t* __restrict__ X, const int32_t* __restrict__ perm, uint16_t* __restrict__ Xp, int K) {
  pdl_wait();  // the previous kernel on the stream may still read Xp
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int m = blockIdx.y;
  const int j0 = 8 * (int)(blockIdx.x * blockDim.x + threadIdx.x);
  if (j0 >= K) return;
  const uint16_t* xr = X + (int64_t)m * K;
  const int4 p0 = *reinterpret_cast<const int4*>(perm + j0);
  const int4 p1 = *reinterpret_cast<const int4*>(perm + j0 + 4);
  const uint4 o = make_uint4((uint32_t)xr[p0.x] | ((uint32_t)xr[p0.y] << 16), (uint32_t)xr[p0.z] | ((uint32_t)xr[p0.w] << 16),
                             (uint32_t)xr[p1.x] | ((uint32_t)xr[p1.y] << 16), (uint32_t)xr[p1.z] | ((uint32_t)xr[p1.w] << 16));
  *reinterpret_cast<uint4*>(Xp + (int64_t)m * K + j0) = o;
}

// The same with the token's row staged in shared memory first (one coalesced read of the row,
// then the permuted reads from shared memory): one CTA per token, K * 2 bytes of smem.
__global__ void __launch_bounds__(256)
    w4_gather_row_kernel(const uint16_t* __restrict__ X, const int32_t* __restrict__ perm, uint16_t* __restrict__ Xp,
                         int K) {
  extern __shared__ __align__(16) uint16_t xrow[];
  pdl_wait();  // the previous kernel on the stream may still read Xp
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int m = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(X + (int64_t)m * K);
  for (int i = threadIdx.x; i < K / 8; i += blockDim.x) reinterpret_cast<uint4*>(xrow)[i] = src[i];
  __syncthreads();
  for (int j0 = 8 * threadIdx.x; j0 < K; j0 += 8 * blockDim.x) {
    const int4 p0 = *reinterpret_cast<const int4*>(perm + j0);
    const int4 p1 = *reinterpret_cast<const int4*>(perm + j0 + 4);
    const uint4 o = make_uint4((uint32_t)xrow[p0.x] | ((uint32_t)xrow[p0.y] << 16),
                               (uint32_t)xrow[p0.z] | ((uint32_t)xrow[p0.w] << 16),
                               (uint32_t)xrow[p1.x] | ((uint32_t)xrow[p1.y] << 16),
                               (uint32_t)xrow[p1.z] | ((uint32_t)xrow[p1.w] << 16));
    *reinterpret_cast<uint4*>(Xp + (int64_t)m * K + j0) = o;
  }
}

constexpr int kGatherRowMaxK = 96 * 1024;  // K * 2 bytes of shared memory per CTA

}  // namespace

int launch_w4_gather(const uint16_t* X, const int32_t* perm, uint16_t* Xp, int M, int K, void* stream) {
  cudaLaunchConfig_t cfg = {};
  // many tokens: stage each row (coalesced); a few tokens: one CTA per row would serialize the
  // row, so many CTAs gather straight from global memory (measured: M = 1 faster, M = 4096 slower)
  if (M > 16 && K <= kGatherRowMaxK) {
    static std::atomic<uint64_t> attr_done{0};  // raised to the largest size, once per device
    const size_t smem = (size_t)K * 2;
    if (smem > 48 * 1024) {
      if (const int e = smem_attr_once(w4_gather_row_kernel, (size_t)kGatherRowMaxK * 2, attr_done)) return e;
    }
    cfg.gridDim = dim3((unsigned)M);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = QLIN_USE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, w4_gather_row_kernel, X, perm, Xp, K);
  }
  cfg.gridDim = dim3((unsigned)((K / 8 + 255) / 256), (unsigned)M);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = QLIN_USE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, w4_gather_kernel, X, perm, Xp, K);
}

int launch_w4_decode(const W4View& v, const uint16_t* X, uint16_t* Y, int M, const Workspace& ws, int grid,
                     void* stream) {
  if (M == 1) return launch_w4_gemv1(v, X, Y, ws, stream);
  // CTAs per SM: up to eight tokens the launch bounds allow four, but a layer under 64 MB of
  // packed weights runs faster with two (fewer CTAs share each split row group, and a CTA's
  // fixed start and finish weigh less).  Same box, us per forward (4 / 2 CTAs per SM): 4096^2
  // M = 2 7.27 / 5.64, M = 4 7.05 / 5.46, M = 8 7.48 / 7.25; 4096 x 11008 M = 4 9.68 / 9.43;
  // 8192^2 M = 4 13.06 / 12.76; 8192 x 28672 (125 MB) M = 4 36.0 / 38.4 the other way.
  const bool small = (int64_t)v.RG * v.G * kW4UnitBytes < (int64_t(64) << 20);
  const int cps = M <= 8 ? (small ? 2 : 4) : QLIN_W4_CPS16;
  grid = (int)std::min<int64_t>((int64_t)v.RG * v.G, (int64_t)std::min(cps, QLIN_DECODE_CPS_MAX) * ws.sms);
  if (M <= 4) return launch_w4_mt<1, 4>(v, X, Y, M, ws, grid, stream);
  if (M <= 8) return launch_w4_mt<1, 0>(v, X, Y, M, ws, grid, stream);
  return launch_w4_mt<2, 0>(v, X, Y, M, ws, grid, stream);
}

}  // namespace qlin

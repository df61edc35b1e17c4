// SmoothQuant W8A8 decode: per-token activation quantization, then an exact integer GEMV.
//
// SmoothQuant page ("Makale Bülteni — SmoothQuant", "İddia ve Gerçeklik: SmoothQuant"):
// X diag(s)^-1 is quantized per token and diag(s) W per output channel to int8, the
// product is accumulated in integers and scaled back.
//
// Act-quant: x' = x * s_inv (fp32), sx = max|x'| / 127 (1 if 0), q = clamp(rint(x'/sx), +-127),
// IEEE division and round-half-to-even, one CTA per token that reads its row once and keeps
// x' in registers (rows up to 32768 wide; a two-pass form for wider ones).  The forward path
// stores the codes as fp16 (exact for |q| <= 127) so the MMA takes them directly: row-major
// for the prefill GEMM's tensor map, K-blocked [K/64][M][72] for the decode GEMV, whose
// X slice per unit is then one bulk copy.
//
// GEMV: Blackwell Ultra's int8 tensor rate is a small fraction of its fp16 rate, so the
// integer product runs on the fp16 MMA instead: int8 codes are exact in fp16, products
// (|q| <= 127^2) are exact in fp32, and any sum of at most 1024 of them stays below 2^24,
// hence exact too.  The kernel drains the fp32 accumulators into int32 every 16 units
// (1024 K) -- the int32 result equals the integer accumulator bit for bit.  Weight bytes are
// stored as u = q + 128 in A-fragment order (a lane's 32 bytes as two 16-byte halves, so the
// warp's loads are contiguous); one byte permute makes fp16 (1024 + u) and one fp16 subtract
// of 1152 leaves q.  Epilogue y = bf16((fp32(acc) * sx_m) * sw_n).
#include "kern_decode_common.cuh"

namespace qlin {
namespace {

#ifndef QLIN_W8_DEC_STAGES
#define QLIN_W8_DEC_STAGES 4
#endif
constexpr int kStagesW8 = QLIN_W8_DEC_STAGES;
constexpr int kXStrideW8 = 72;  // staged qx row: 64 fp16 + 8 pad

// Where the fp16 code of (token m, channel k) goes.  blk == 0: row-major [M][K] (the prefill
// GEMM's TMA map).  blk == M: blocked for the decode GEMV, [K/64][M][kXStrideW8], so that one
// bulk copy moves a 64-wide K block of every token into the staged layout (pad not written).
__device__ __forceinline__ int64_t q16_offset(int m, int k, int K, int blk) {
  if (blk == 0) return (int64_t)m * K + k;
  return ((int64_t)(k >> 6) * blk + m) * kXStrideW8 + (k & 63);
}

template <bool F16OUT>
__global__ void __launch_bounds__(256)
    w8_act_quant_kernel(const uint16_t* __restrict__ X, const float* __restrict__ s_inv, int K,
                        int8_t* __restrict__ q8, uint16_t* __restrict__ q16, float* __restrict__ sx,
                        int32_t* __restrict__ kbound, int blk) {
  __shared__ float red[8];
  __shared__ float scale_sh;
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int m = blockIdx.x;
  const uint16_t* xr = X + (int64_t)m * K;
  float amax = 0.f;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const uint4 xv = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = __uint_as_float(((xw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
      amax = fmaxf(amax, fabsf(__fmul_rn(x, s_inv[k + e])));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) a = fmaxf(a, red[i]);
    const float sc = a == 0.f ? 1.f : __fdiv_rn(a, 127.f);
    scale_sh = sc;
    sx[m] = sc;
  }
  __syncthreads();
  const float sc = scale_sh;
  for (int k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
    const uint4 xv = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    int qv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = __uint_as_float(((xw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
      int q = __float2int_rn(__fdiv_rn(__fmul_rn(x, s_inv[k + e]), sc));
      qv[e] = q < -127 ? -127 : (q > 127 ? 127 : q);
    }
    if (kbound) {
      // sum q^2 of this token's 64-wide k-block (8 threads of 8 codes), max into its tile's bound
      int l2 = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) l2 += qv[e] * qv[e];
      // K is a multiple of 64, so the 8 lanes of a k-block are in the loop together (a warp's
      // tail may not be)
      const unsigned am = __activemask();
      l2 += __shfl_xor_sync(am, l2, 1);
      l2 += __shfl_xor_sync(am, l2, 2);
      l2 += __shfl_xor_sync(am, l2, 4);
      if ((threadIdx.x & 7) == 0) atomicMax(kbound + (int64_t)(m >> 8) * (K / 64) + k / 64, l2);
    }
    if constexpr (F16OUT) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 h = __halves2half2(__int2half_rn(qv[2 * e]), __int2half_rn(qv[2 * e + 1]));
        o[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(q16 + q16_offset(m, k, K, blk)) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo |= (uint32_t)(uint8_t)(int8_t)qv[e] << (8 * e);
        hi |= (uint32_t)(uint8_t)(int8_t)qv[4 + e] << (8 * e);
      }
      *reinterpret_cast<uint2*>(q8 + (int64_t)m * K + k) = make_uint2(lo, hi);
    }
  }
}

// The same quantization in a single read: one CTA of kAqThreads threads per token, each
// thread holding R chunks of 8 scaled activations x' in registers between the row maximum and
// the rounding (rows up to kAqThreads * 8 * R wide).  The arithmetic is the two-pass kernel's,
// operation for operation, so the codes and scales are the same bits.
constexpr int kAqThreads = 512;

template <bool F16OUT, int R>
__global__ void __launch_bounds__(kAqThreads)
    w8_act_quant_reg_kernel(const uint16_t* __restrict__ X, const float* __restrict__ s_inv, int K,
                            int8_t* __restrict__ q8, uint16_t* __restrict__ q16, float* __restrict__ sx,
                            int32_t* __restrict__ kbound, int blk) {
  __shared__ float red[kAqThreads / 32];
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int m = blockIdx.x, lane = threadIdx.x & 31;
  const uint16_t* xr = X + (int64_t)m * K;
  const int nc = K >> 3;  // chunks of 8
  float xs[R][8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int c = threadIdx.x + i * kAqThreads;
    if (c < nc) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xr + 8 * c);
      const float4 s0 = *reinterpret_cast<const float4*>(s_inv + 8 * c);
      const float4 s1 = *reinterpret_cast<const float4*>(s_inv + 8 * c + 4);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = __uint_as_float((e & 1) ? (xw[e >> 1] & 0xFFFF0000u) : (xw[e >> 1] << 16));
        xs[i][e] = __fmul_rn(x, sv[e]);
        amax = fmaxf(amax, fabsf(xs[i][e]));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) xs[i][e] = 0.f;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  float a = red[0];
#pragma unroll
  for (int i = 1; i < kAqThreads / 32; ++i) a = fmaxf(a, red[i]);
  const float sc = a == 0.f ? 1.f : __fdiv_rn(a, 127.f);
  if (threadIdx.x == 0) sx[m] = sc;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int c = threadIdx.x + i * kAqThreads;
    const bool valid = c < nc;
    int qv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int q = valid ? __float2int_rn(__fdiv_rn(xs[i][e], sc)) : 0;
      qv[e] = q < -127 ? -127 : (q > 127 ? 127 : q);
    }
    if (kbound) {
      // sum q^2 over a 64-wide k-block: 8 consecutive chunks are 8 consecutive lanes, all valid
      // or all past the row (K is a multiple of 64)
      int l2 = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) l2 += qv[e] * qv[e];
      l2 += __shfl_xor_sync(0xffffffffu, l2, 1);
      l2 += __shfl_xor_sync(0xffffffffu, l2, 2);
      l2 += __shfl_xor_sync(0xffffffffu, l2, 4);
      if (valid && (lane & 7) == 0) atomicMax(kbound + (int64_t)(m >> 8) * (K / 64) + c / 8, l2);
    }
    if (!valid) continue;
    if constexpr (F16OUT) {
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __half2 h = __halves2half2(__int2half_rn(qv[2 * e]), __int2half_rn(qv[2 * e + 1]));
        o[e] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(q16 + q16_offset(m, 8 * c, K, blk)) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo |= (uint32_t)(uint8_t)(int8_t)qv[e] << (8 * e);
        hi |= (uint32_t)(uint8_t)(int8_t)qv[4 + e] << (8 * e);
      }
      *reinterpret_cast<uint2*>(q8 + (int64_t)m * K + 8 * c) = make_uint2(lo, hi);
    }
  }
}

template <int MT>
struct W8Smem {
  __align__(16) uint8_t unit[kStagesW8][kW8UnitBytes];
  __align__(16) uint16_t x[kStagesW8][8 * MT][kXStrideW8];
  uint64_t full[kStagesW8];
  uint64_t empty[kStagesW8];
  uint64_t cons_bar;
  int flags[2];
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

template <int MT>
__global__ void __launch_bounds__(160, MT == 1 ? 4 : 3)
    w8_decode_kernel(W8View v, const uint16_t* __restrict__ q16, const float* __restrict__ sx,
                     uint16_t* __restrict__ Y, int32_t* __restrict__ acc_out, int M, Workspace ws) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  W8Smem<MT>& sm = *reinterpret_cast<W8Smem<MT>*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t grid = gridDim.x, cta = blockIdx.x;
  const int64_t KB = v.KB, U = (int64_t)v.RG * KB;
  const int64_t u0 = split_start(cta, U, grid), u1 = split_start(cta + 1, U, grid);
  const int n_units = (int)(u1 - u0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesW8; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 4);
    }
    mbar_init(&sm.cons_bar, 128);
    fence_mbar_init();
    pdl_launch_dependents();
  }
  {
    uint32_t* xz = reinterpret_cast<uint32_t*>(&sm.x[0][0][0]);
    for (int i = threadIdx.x; i < kStagesW8 * 8 * MT * kXStrideW8 / 2; i += blockDim.x) xz[i] = 0u;
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == 4) {
    if (lane != 0) return;
    // the codes are blocked [K/64][M][kXStrideW8]: a unit's X slice is one contiguous copy
    const uint32_t xbytes = (uint32_t)M * kXStrideW8 * 2;
    const uint32_t tx = kW8UnitBytes + xbytes;
    int kx = (int)(u0 % KB);  // K block of the next X slice (units are issued in order)
    auto load_x = [&](int s) {
      bulk_g2s(&sm.x[s][0][0], q16 + (int64_t)kx * M * kXStrideW8, xbytes, &sm.full[s]);
      if (++kx == (int)KB) kx = 0;
    };
    const int pro = n_units < kStagesW8 ? n_units : kStagesW8;
    for (int i = 0; i < pro; ++i) {
      mbar_arrive_expect_tx(&sm.full[i], tx);
      bulk_g2s(sm.unit[i], v.units + (u0 + i) * (int64_t)kW8UnitBytes, kW8UnitBytes, &sm.full[i]);
    }
    pdl_wait();  // the activation codes come from the act-quant kernel
    for (int i = 0; i < pro; ++i) load_x(i);
    for (int i = kStagesW8; i < n_units; ++i) {
      const int s = i % kStagesW8;
      const uint32_t ph = (uint32_t)(i / kStagesW8) & 1u;
      if (!mbar_wait(&sm.empty[s], ph ^ 1u, ws.status)) return;
      mbar_arrive_expect_tx(&sm.full[s], tx);
      bulk_g2s(sm.unit[s], v.units + (u0 + i) * (int64_t)kW8UnitBytes, kW8UnitBytes, &sm.full[s]);
      load_x(s);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = lane >> 2, t = lane & 3;
  ConsumerSync cs{&sm.cons_bar, 0u, ws.status};
  int32_t iacc[MT][4];
  float c[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      iacc[mt][i] = 0;
      c[mt][i] = 0.f;
    }
  int since_drain = 0;
  auto drain = [&]() {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        iacc[mt][i] += __float2int_rn(c[mt][i]);
        c[mt][i] = 0.f;
      }
    since_drain = 0;
  };
  int64_t cur_rg = u0 / KB;
  UnitCursor cur{cur_rg, (int)(u0 - cur_rg * KB), (int)KB};

  int idx[MT * 4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = warp * 16 + g + ((i & 2) ? 8 : 0);
      const int m = 2 * t + (i & 1) + 8 * mt;
      idx[mt * 4 + i] = (m < M) ? r * 16 + m : -1;
    }
  auto done = [&](int64_t rg, const int (&out)[MT * 4]) {
#pragma unroll
    for (int j = 0; j < MT * 4; ++j) {
      if (idx[j] < 0) continue;
      const int64_t n = rg * kRowGroup + idx[j] / 16;
      const int m = idx[j] % 16;
      if (n >= v.N) continue;
      if (acc_out) {
        acc_out[(int64_t)m * v.N + n] = out[j];
      } else {
        const float y = __fmul_rn(__fmul_rn(__int2float_rn(out[j]), sx[m]), v.sw[n]);
        Y[(int64_t)m * v.N + n] = f2bf(y);
      }
    }
  };
  RowGroupFinisher<int, MT * 4> fin(KB, U, grid, cta, ws.partials, ws.counters);
  auto flush = [&](int64_t rg) {
    drain();
    int vals[MT * 4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) vals[mt * 4 + i] = iacc[mt][i];
    fin.stage(rg, vals, idx, done);
  };

  // the previous kernel on the stream may still read this launch's outputs or workspace
  pdl_wait();
  for (int i = 0; i < n_units; ++i) {
    const int s = i % kStagesW8;
    const uint32_t ph = (uint32_t)(i / kStagesW8) & 1u;
    const int64_t rg = cur.rg;
    cur.next();
    if (rg != cur_rg) {
      flush(cur_rg);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int q = 0; q < 4; ++q) iacc[mt][q] = 0;
      cur_rg = rg;
    }
    if (!mbar_wait(&sm.full[s], ph, ws.status)) return;
    // the lane's 8 words as two halves, each a contiguous 512 bytes across the warp
    const uint4 w01 = *reinterpret_cast<const uint4*>(sm.unit[s] + ((warp * 2 + 0) * 32 + lane) * 16);
    const uint4 w23 = *reinterpret_cast<const uint4*>(sm.unit[s] + ((warp * 2 + 1) * 32 + lane) * 16);
    const uint32_t words[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
    const uint32_t magic = 0x64646464u, off = 0x64806480u;  // fp16 1152 = 1024 + 128
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t a[4];
      a[0] = f16x2_sub(prmt(words[2 * j], magic, 0x5140u), off);
      a[1] = f16x2_sub(prmt(words[2 * j], magic, 0x5342u), off);
      a[2] = f16x2_sub(prmt(words[2 * j + 1], magic, 0x5140u), off);
      a[3] = f16x2_sub(prmt(words[2 * j + 1], magic, 0x5342u), off);
      const int kk = 16 * j + 2 * t;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint16_t* xr = &sm.x[s][g + 8 * mt][0];
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xr + kk);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(xr + kk + 8);
        mma_f16(c[mt], a, b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    if (++since_drain == 16) drain();
  }
  if (n_units > 0) {
    flush(cur_rg);
    fin.finish(M, cs, sm.flags, [&](int64_t rg, int e, int val) {
      const int64_t n = rg * kRowGroup + e / 16;
      const int m = e % 16;
      if (n >= v.N) return;
      if (acc_out) {
        acc_out[(int64_t)m * v.N + n] = val;
      } else {
        Y[(int64_t)m * v.N + n] = f2bf(__fmul_rn(__fmul_rn(__int2float_rn(val), sx[m]), v.sw[n]));
      }
    });
  }
}

template <int MT>
int launch_w8_mt(const W8View& v, const uint16_t* q16, const float* sx, uint16_t* Y, int32_t* acc, int M,
                 const Workspace& ws, int grid, void* stream) {
  const size_t smem = sizeof(W8Smem<MT>);
  static std::atomic<uint64_t> attr_done{0};
  if (const int e = smem_attr_once(w8_decode_kernel<MT>, smem, attr_done)) return e;
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
  return (int)cudaLaunchKernelEx(&cfg, w8_decode_kernel<MT>, v, q16, sx, Y, acc, M, ws);
}

template <bool F16>
int launch_aq(const W8View& v, const uint16_t* X, int8_t* q8, uint16_t* q16, float* sx, int32_t* kbound, int M,
              int blk, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(kAqThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = QLIN_USE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int chunks = v.K / 8;
  if (chunks <= kAqThreads)
    return (int)cudaLaunchKernelEx(&cfg, w8_act_quant_reg_kernel<F16, 1>, X, v.s_inv, v.K, q8, q16, sx, kbound, blk);
  if (chunks <= 2 * kAqThreads)
    return (int)cudaLaunchKernelEx(&cfg, w8_act_quant_reg_kernel<F16, 2>, X, v.s_inv, v.K, q8, q16, sx, kbound, blk);
  if (chunks <= 4 * kAqThreads)
    return (int)cudaLaunchKernelEx(&cfg, w8_act_quant_reg_kernel<F16, 4>, X, v.s_inv, v.K, q8, q16, sx, kbound, blk);
  if (chunks <= 8 * kAqThreads)
    return (int)cudaLaunchKernelEx(&cfg, w8_act_quant_reg_kernel<F16, 8>, X, v.s_inv, v.K, q8, q16, sx, kbound, blk);
  cfg.blockDim = dim3(256);  // wider rows: the two-pass kernel
  return (int)cudaLaunchKernelEx(&cfg, w8_act_quant_kernel<F16>, X, v.s_inv, v.K, q8, q16, sx, kbound, blk);
}

}  // namespace

int launch_w8_act_quant(const W8View& v, const uint16_t* X, int8_t* qx, float* sx, int M, void* stream) {
  return launch_aq<false>(v, X, qx, nullptr, sx, nullptr, M, 0, stream);
}

int launch_w8_act_quant_f16(const W8View& v, const uint16_t* X, uint16_t* q16, float* sx, int32_t* kbound, int M,
                            bool blocked, void* stream) {
  return launch_aq<true>(v, X, nullptr, q16, sx, kbound, M, blocked ? M : 0, stream);
}

int launch_w8_decode(const W8View& v, const uint16_t* q16, const float* sx, uint16_t* Y, int32_t* acc_out, int M,
                     const Workspace& ws, int grid, void* stream) {
  const int64_t U = (int64_t)v.RG * v.KB;
  // up to eight tokens: four CTAs per SM, three for a layer under 24 MB of packed weights (same
  // box, us per forward, four / three: 4096^2 M = 2 10.21 / 9.88, M = 4 10.70 / 10.26, M = 8
  // 11.99 / 11.16; 8192^2 and the 70B-class layer measured the other way)
  const int cps8 = U * kW8UnitBytes < (int64_t(24) << 20) ? 3 : 4;
  if (M <= 8) return launch_w8_mt<1>(v, q16, sx, Y, acc_out, M, ws, (int)std::min<int64_t>(U, (int64_t)std::min(cps8, QLIN_DECODE_CPS_MAX) * ws.sms), stream);
  return launch_w8_mt<2>(v, q16, sx, Y, acc_out, M, ws, (int)std::min<int64_t>(U, (int64_t)std::min(3, QLIN_DECODE_CPS_MAX) * ws.sms), stream);
}

}  // namespace qlin

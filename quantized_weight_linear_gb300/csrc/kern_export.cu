// Decoders of the device weight images back to dense form (test and inspection path), and
// the device-side wait-limit test hook.
//
// The decoders read the same unit layouts the forward kernels stream and recompute each
// weight with the formats' arithmetic in fp32, round-to-nearest and no fused multiply-add:
//   W4G128: w = (q - z) * s
//   SPQR:   s^ = (qs - zs) * ss, z^ = (qz - zz) * sz, D = (q - z^) * s^, W = D (+ fp16 outlier)
//   W8A8:   qw = u - 128
// so the result must equal the canonical arrays' dequantization bit for bit.
#include "kern_common.cuh"

namespace qlin {
namespace {

__global__ void w4_dequant_kernel(W4View v, float* __restrict__ out) {
  const int64_t total = (int64_t)v.N * v.K;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = idx / v.K;
    const int k = (int)(idx % v.K);
    const int64_t rg = n / kRowGroup;
    const int rt = (int)((n % kRowGroup) / 16), r = (int)(n % 16);
    const int grp = k / kW4Group, kb = (k % kW4Group) / 64, kk = k % 64, j = kk / 16, kr = kk % 16;
    const int g = r & 7, rowhi = r >> 3;
    const int khi = kr >= 8 ? 1 : 0;
    const int t = (kr - 8 * khi) >> 1, kodd = kr & 1;
    const uint8_t* unit = v.units + (rg * v.G + grp) * (int64_t)kW4UnitBytes;
    const uint32_t w = reinterpret_cast<const uint32_t*>(unit)[((rt * 2 + kb) * 32 + 4 * g + t) * 4 + j];
    const int nib = rowhi + 2 * khi + 4 * kodd;
    const uint32_t q = (w >> (4 * nib)) & 15u;
    const uint32_t sz = reinterpret_cast<const uint32_t*>(unit + kW4CodeBytes)[rt * 16 + r];
    const float s = h2f_dev((uint16_t)(sz & 0xFFFFu)), z = h2f_dev((uint16_t)(sz >> 16));
    out[idx] = __fmul_rn(__fsub_rn((float)q, z), s);
  }
}

// 3-bit code of (row r in tile, k in block) from a block's lane words
__device__ __forceinline__ uint32_t spqr_code_at(const uint32_t* blockwords, int r, int kblk) {
  const int gb = kblk / 16, e = kblk % 16, j = e >> 1, half = e & 1;
  const int g = r & 7;
  const int ra = (r >> 3) | ((gb >= 4) ? 2 : 0);  // A register index
  const int t = gb & 3;
  const uint32_t* w = blockwords + (4 * g + t) * 6;
  if (j <= 4) {
    const int i = 4 * j + ra;
    if (i < 18) {
      const int f = (i % 3) * 2;
      return (w[i / 3] >> (3 * f + 16 * half)) & 7u;
    }
    const int b = 3 * (i - 18);
    const int bit = half ? 31 : 15;
    return ((w[b] >> bit) & 1u) | (((w[b + 1] >> bit) & 1u) << 1) | (((w[b + 2] >> bit) & 1u) << 2);
  }
  const int i = 4 * (j - 5) + ra;
  const int f = (i % 2) * 2 + 1;
  return (w[i / 2] >> (3 * f + 16 * half)) & 7u;
}

__device__ __forceinline__ uint32_t spqr_qsqz_at(const uint8_t* area, int r, int gb) {
  const int lane = 4 * (r & 7) + (gb >> 1);
  const int i = ((r >> 3) << 1) | (gb & 1);
  const int bit = 24 * lane + 6 * i;
  uint32_t v = 0;
  for (int b = 0; b < 6; ++b) v |= (uint32_t)((area[(bit + b) >> 3] >> ((bit + b) & 7)) & 1u) << b;
  return v;
}

__global__ void spqr_dense_kernel(SpqrView v, float* __restrict__ out) {
  const int64_t total = (int64_t)v.N * v.K;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = idx / v.K;
    const int k = (int)(idx % v.K);
    const int64_t rg = n / kRowGroup;
    const int rt = (int)((n % kRowGroup) / 16), r = (int)(n % 16);
    const int sg = k / kSpqrSuper, blk = (k % kSpqrSuper) / 128, kblk = k % 128;
    const uint8_t* unit = v.units + (rg * v.S + sg) * (int64_t)kSpqrUnitBytes;
    const uint32_t* words = reinterpret_cast<const uint32_t*>(unit) + (rt * 2 + blk) * 32 * 6;
    const uint32_t q = spqr_code_at(words, r, kblk);
    const uint32_t e = spqr_qsqz_at(unit + kSpqrCodeBytes + (rt * 2 + blk) * 96, r, kblk / 16);
    const uint16_t* st = reinterpret_cast<const uint16_t*>(unit + kSpqrCodeBytes + kSpqrQsqzBytes) + (rt * 16 + r) * 4;
    const float ss = h2f_dev(st[0]), zs = h2f_dev(st[1]), sz = h2f_dev(st[2]), zz = h2f_dev(st[3]);
    const float sh = __fmul_rn(__fsub_rn((float)(e & 7u), zs), ss);
    const float zh = __fmul_rn(__fsub_rn((float)(e >> 3), zz), sz);
    out[idx] = __fmul_rn(__fsub_rn((float)q, zh), sh);
  }
}

__global__ void spqr_outlier_kernel(SpqrView v, float* __restrict__ out) {
  const int64_t buckets = (int64_t)v.RG * v.S * 4;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < buckets; b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t unit = b / 4;
    const int rt = (int)(b % 4);
    const int64_t rg = unit / v.S, sg = unit % v.S;
    for (uint32_t p = v.offs[b]; p < v.offs[b + 1]; ++p) {
      const uint32_t e = v.ents[p];
      const int64_t n = rg * kRowGroup + rt * 16 + (e & 15u);
      const int64_t k = sg * kSpqrSuper + ((e >> 4) & 255u);
      float* o = out + n * v.K + k;
      *o = __fadd_rn(*o, h2f_dev((uint16_t)(e >> 16)));
    }
  }
}

__global__ void w8_export_kernel(W8View v, int8_t* __restrict__ out) {
  const int64_t total = (int64_t)v.N * v.K;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = idx / v.K;
    const int k = (int)(idx % v.K);
    const int64_t rg = n / kRowGroup;
    const int rt = (int)((n % kRowGroup) / 16), r = (int)(n % 16);
    const int kb = k / kW8Block, kk = k % kW8Block, j = kk / 16, kr = kk % 16;
    const int g = r & 7, rowhi = r >> 3, khi = kr >= 8 ? 1 : 0, t = (kr - 8 * khi) >> 1, kodd = kr & 1;
    const uint8_t* unit = v.units + (rg * v.KB + kb) * (int64_t)kW8UnitBytes;
    const int lane = 4 * g + t;  // word 2j + khi of the lane: half j / 2, bytes (j % 2) * 8 + khi * 4 ..
    const uint8_t u = unit[((rt * 2 + (j >> 1)) * 32 + lane) * 16 + (j & 1) * 8 + khi * 4 + rowhi * 2 + kodd];
    out[idx] = (int8_t)((int)u - 128);
  }
}

__global__ void wait_timeout_kernel(int32_t* status, int limit_us) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on this barrier: the bounded wait must give up and report it
    mbar_wait(&bar, 0, status, (uint64_t)limit_us * 1000ull);
  }
}

int grid_for(int64_t total) {
  int64_t b = (total + 255) / 256;
  if (b > 4096) b = 4096;
  if (b < 1) b = 1;
  return (int)b;
}

}  // namespace

int launch_w4_dequant(const W4View& v, float* out, void* stream) {
  w4_dequant_kernel<<<grid_for((int64_t)v.N * v.K), 256, 0, (cudaStream_t)stream>>>(v, out);
  return (int)cudaGetLastError();
}

int launch_spqr_dequant(const SpqrView& v, float* out, void* stream) {
  spqr_dense_kernel<<<grid_for((int64_t)v.N * v.K), 256, 0, (cudaStream_t)stream>>>(v, out);
  spqr_outlier_kernel<<<grid_for((int64_t)v.RG * v.S * 4), 256, 0, (cudaStream_t)stream>>>(v, out);
  return (int)cudaGetLastError();
}

int launch_w8_export(const W8View& v, int8_t* out, void* stream) {
  w8_export_kernel<<<grid_for((int64_t)v.N * v.K), 256, 0, (cudaStream_t)stream>>>(v, out);
  return (int)cudaGetLastError();
}

int launch_debug_wait_timeout(int32_t* status, int limit_us, void* stream) {
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, limit_us);
  return (int)cudaGetLastError();
}

}  // namespace qlin

// Device helpers shared by the libqlin kernels (sm_103a).
//
// * mbarrier waits are bounded in wall time (%globaltimer, 2 s by default): a waiter that
//   runs out records kStatusTimeout in the workspace status word and gives up, so a broken
//   pipeline ends with an error the host can read instead of a hung GPU.
// * Bulk copies use the non-tensor cp.async.bulk (TMA engine, 16-byte granularity) with
//   mbarrier transaction counts.
// * Launches use programmatic dependent launch: a kernel may start streaming weights while
//   the previous kernel on the stream drains, and waits (griddepcontrol.wait) before it
//   touches activations, outputs or workspace.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "qlin_internal.h"

namespace qlin {


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 2D tiled TMA load of box (x, y) of `map` into shared memory (128-byte aligned destination),
// completing on `bar`'s transaction count
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// The driver's tensor-map encoder (looked up once through the runtime)
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Map of the decode kernels' activations X [M][K] bf16 (row-major): boxes of box_k channels of
// all M tokens, unswizzled, so one copy lands as M rows of box_k elements.  Channels past K
// read as zero.  Returns false if the encoder is missing or refuses the shape.
inline bool encode_decode_x_map(CUtensorMap* map, const void* X, int64_t K, int M, int box_k) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_k, (cuuint32_t)M};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device): the attribute is per device, so a process driving several GPUs needs it on
// each.  `done` holds one bit per device id < 64 (larger ids set it on every call).
template <typename Kernel>
inline int smem_attr_once(Kernel* kernel, size_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return 0;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return (int)e;
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return 0;
}

// Dynamic shared memory rounded up to a 128-byte boundary (the launch adds 128 bytes)
__device__ __forceinline__ uint8_t* smem_align128(uint8_t* raw) {
  return raw + ((128u - (smem_u32(raw) & 127u)) & 127u);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with an explicit suspend-time hint (ns), so one poll never sleeps longer than that
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on the phase with the given parity: gives up after `limit_ns` of wall time
// (default 2 s), records the timeout in *status (if non-null) and returns false.
// QLIN_WAIT_HINT_NS: suspend-time hint of each poll (0 = the hardware's default limit).
#ifndef QLIN_WAIT_HINT_NS
#define QLIN_WAIT_HINT_NS 0
#endif
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (QLIN_WAIT_HINT_NS > 0 ? mbar_try_wait_hint(bar, parity, QLIN_WAIT_HINT_NS) : mbar_try_wait(bar, parity))
      return true;
    if (global_ns() - t0 > limit_ns) break;
  }
  if (status) atomicExch(status, kStatusTimeout);
  return false;
}

// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// 16-byte load through L2 only (data written by other SMs in this launch)
__device__ __forceinline__ void ldcg4(const float* p, float (&v)[4]) {
  const float4 q = __ldcg(reinterpret_cast<const float4*>(p));
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void ldcg4(const int* p, int (&v)[4]) {
  const int4 q = __ldcg(reinterpret_cast<const int4*>(p));
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}

// Upper bound on the CTAs per SM the decode launches use (their occupancy allows up to 4).
#ifndef QLIN_DECODE_CPS_MAX
#define QLIN_DECODE_CPS_MAX 4
#endif

// Programmatic dependent launch for the decode and prefill kernels (1 = on).
#ifndef QLIN_USE_PDL
#define QLIN_USE_PDL 1
#endif

// global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// barrier `id` (1..15) over `threads` threads (a multiple of 32), every one of which must
// reach it
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_4(float& d0, float& d1, float& d2, float& d3, const uint32_t (&a)[4],
                                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A(16x16 f16) * B(16x8 f16), fp32 accumulate
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  return (a & mask) | orv;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t b) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 r = __hadd2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
  __nv_bfloat162 z = *reinterpret_cast<__nv_bfloat162*>(&c);
  __nv_bfloat162 r = __hfma2(x, y, z);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  __half2 y = *reinterpret_cast<__half2*>(&b);
  __half2 r = __hsub2(x, y);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint16_t f2bf(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float bf2f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

__device__ __forceinline__ float h2f_dev(uint16_t v) { return __half2float(__ushort_as_half(v)); }

// Static split of `units` work units over `grid` CTAs: CTA c owns [start(c), start(c+1)).
__device__ __forceinline__ int64_t split_start(int64_t c, int64_t units, int64_t grid) {
  return c * units / grid;
}
// The CTA whose range contains unit u.
__device__ __forceinline__ int64_t split_owner(int64_t u, int64_t units, int64_t grid) {
  return ((u + 1) * grid - 1) / units;
}

// Cross-CTA completion of a row group split over several CTAs.  Every contributor stores
// its partial sums (64 rows x 16 tokens, fp32 or int32 bits) into its slot
// partials[(cta * 2 + side) * 1024 ...], then counts itself on counters[rg]; the last one
// sums all slots in CTA order (deterministic) and writes the row group.  The counter is
// reset to 0 by the last contributor so the next forward starts clean.
struct SplitInfo {
  int64_t first_cta, last_cta;
};

__device__ __forceinline__ SplitInfo split_info(int64_t rg, int64_t per_rg, int64_t units, int64_t grid) {
  SplitInfo s;
  s.first_cta = split_owner(rg * per_rg, units, grid);
  s.last_cta = split_owner(rg * per_rg + per_rg - 1, units, grid);
  return s;
}

__device__ __forceinline__ int split_side(int64_t cta, int64_t rg, int64_t per_rg, int64_t units, int64_t grid) {
  const int64_t first_rg = split_start(cta, units, grid) / per_rg;
  return rg == first_rg ? 0 : 1;
}

}  // namespace qlin

// Pieces shared by the decode (M <= 16) GEMV kernels: the consumer-group barrier and the
// split-row-group completion protocol.
#pragma once
#include "kern_common.cuh"

namespace qlin {

// A reusable barrier for the 128 consumer threads (4 warps) built on an mbarrier, so that
// its wait is bounded like every other wait in the kernels.
struct ConsumerSync {
  uint64_t* bar;
  uint32_t phase;
  int32_t* status;
  __device__ __forceinline__ bool sync() {
    mbar_arrive(bar);
    bool ok = mbar_wait(bar, phase, status);
    phase ^= 1u;
    return ok;
  }
};

// Completion of one row group (64 rows x up to 16 tokens).  `vals[i]` is the value of
// entry idx[i] = row_in_group * 16 + token held by this thread (nv entries, invalid ones
// flagged by idx < 0).  T is float or int (integer sums are exact).
// Returns false if a bounded wait gave up.  If the row group belongs to this CTA alone,
// `done` is called with the finished values straight away; otherwise the values go to
// the CTA's slot and the last contributor calls `done` with the sums.
template <typename T, int NV, typename Done>
__device__ __forceinline__ bool finish_row_group(int64_t rg, int64_t per_rg, int64_t units, int64_t grid,
                                                 int64_t cta, const T (&vals)[NV], const int (&idx)[NV],
                                                 const Workspace& ws, ConsumerSync& cs, int* flag,
                                                 Done done) {
  const SplitInfo si = split_info(rg, per_rg, units, grid);
  if (si.first_cta == si.last_cta) {
    done(vals);
    return true;
  }
  const int side = split_side(cta, rg, per_rg, units, grid);
  T* slot = reinterpret_cast<T*>(ws.partials) + (cta * 2 + side) * (kRowGroup * 16);
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (idx[i] >= 0) slot[idx[i]] = vals[i];
  __threadfence();
  if (!cs.sync()) return false;
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(&ws.counters[rg], 1u);
    *flag = (old == (unsigned)(si.last_cta - si.first_cta)) ? 1 : 0;
  }
  if (!cs.sync()) return false;
  if (*flag) {
    __threadfence();
    T sum[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) sum[i] = T(0);
    for (int64_t c = si.first_cta; c <= si.last_cta; ++c) {
      const int sd = split_side(c, rg, per_rg, units, grid);
      const T* sl = reinterpret_cast<const T*>(ws.partials) + (c * 2 + sd) * (kRowGroup * 16);
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (idx[i] >= 0) sum[i] += __ldcg(sl + idx[i]);
    }
    done(sum);
    if (threadIdx.x == 0) ws.counters[rg] = 0u;
  }
  return cs.sync();
}

}  // namespace qlin

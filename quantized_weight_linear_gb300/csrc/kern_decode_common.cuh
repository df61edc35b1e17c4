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

// Completion of row groups (64 rows x up to 16 tokens) whose units are split between CTAs.
// A CTA's contiguous unit range can split at most two row groups (its first and its last);
// every other row group it touches is whole and is written straight away.
//
// stage(): a whole row group goes to `done` at once; a split one is stored into this CTA's
// partial slot (plain stores, nothing waits).  finish(), once at the end of the range: one
// fence, one arrival per split row group on its counter, and the last contributor sums all
// slots in CTA order (deterministic) and hands the sums to `done`, then resets the counter
// for the next forward.  So no consumer ever stalls on another CTA in the middle of its
// stream.  `vals[i]` is the value of entry idx[i] = row_in_group * 16 + token (idx < 0:
// unused).  T is float or int (integer sums are exact).
template <typename T, int NV>
struct RowGroupFinisher {
  int64_t per_rg, units, grid, cta;
  const Workspace* ws;
  int64_t pend[2];
  int npend;

  __device__ __forceinline__ RowGroupFinisher(int64_t per_rg_, int64_t units_, int64_t grid_, int64_t cta_,
                                              const Workspace* ws_)
      : per_rg(per_rg_), units(units_), grid(grid_), cta(cta_), ws(ws_), npend(0) {}

  template <typename Done>
  __device__ __forceinline__ void stage(int64_t rg, const T (&vals)[NV], const int (&idx)[NV], Done done) {
    const SplitInfo si = split_info(rg, per_rg, units, grid);
    if (si.first_cta == si.last_cta) {
      done(rg, vals);
      return;
    }
    const int side = split_side(cta, rg, per_rg, units, grid);
    T* slot = reinterpret_cast<T*>(ws->partials) + (cta * 2 + side) * (kRowGroup * 16);
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (idx[i] >= 0) slot[idx[i]] = vals[i];
    if (npend < 2) pend[npend++] = rg;
  }

  // Returns false if a bounded wait gave up.  `flags` is a 2-int shared array.  The last
  // contributor reduces with all 128 consumer threads: thread j takes entries j, j + 128, ...
  // of the 64 x M outputs and loads the contributors' slots eight at a time (one round trip
  // per eight CTAs), summing them in CTA order.  `put(rg, entry, value)` stores one output.
  template <typename Put>
  __device__ __forceinline__ bool finish(int M, ConsumerSync& cs, int* flags, Put put) {
    if (npend == 0) return true;  // uniform: every consumer thread walks the same row groups
    __threadfence();
    if (!cs.sync()) return false;
    if (threadIdx.x == 0) {
      for (int p = 0; p < npend; ++p) {
        const SplitInfo si = split_info(pend[p], per_rg, units, grid);
        const unsigned old = atomicAdd(&ws->counters[pend[p]], 1u);
        flags[p] = (old == (unsigned)(si.last_cta - si.first_cta)) ? 1 : 0;
      }
    }
    if (!cs.sync()) return false;
    for (int p = 0; p < npend; ++p) {
      if (!flags[p]) continue;
      __threadfence();
      const int64_t rg = pend[p];
      const SplitInfo si = split_info(rg, per_rg, units, grid);
      const T* base = reinterpret_cast<const T*>(ws->partials);
      for (int lin = threadIdx.x; lin < kRowGroup * M; lin += 128) {
        const int e = (lin / M) * 16 + lin % M;
        T s = T(0);
        for (int64_t c0 = si.first_cta; c0 <= si.last_cta; c0 += 8) {
          T v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int64_t c = c0 + u;
            v[u] = T(0);
            if (c <= si.last_cta)
              v[u] = __ldcg(base + (c * 2 + split_side(c, rg, per_rg, units, grid)) * (kRowGroup * 16) + e);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) s += v[u];
        }
        put(rg, e, s);
      }
      if (threadIdx.x == 0) ws->counters[rg] = 0u;
    }
    return true;
  }
};

}  // namespace qlin

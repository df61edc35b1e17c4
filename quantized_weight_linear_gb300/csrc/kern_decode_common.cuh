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

// Row group of the current unit in a CTA's contiguous range, advanced without a division.
struct UnitCursor {
  int64_t rg;
  int k;    // unit index inside the row group
  int per;  // units per row group
  __device__ __forceinline__ void next() {
    if (++k == per) {
      k = 0;
      ++rg;
    }
  }
};

// Completion of row groups (64 rows x up to 16 tokens) whose units are split between CTAs.
// A CTA's contiguous unit range can share at most two row groups with other CTAs (its first
// and its last); every other row group it touches is whole and is written straight away.
// Which of the two are shared, by how many CTAs, and where the first contributor keeps its
// partial sums is worked out once, when the finisher is built (before the stream starts).
//
// stage(): a whole row group goes to `done` at once; a shared one is stored into this CTA's
// partial slot (plain stores, nothing waits).  finish(), once at the end of the range: one
// arrival per shared row group on its counter, and the CTA that arrives last sums all slots
// in CTA order (deterministic) and hands the sums to `put`, then resets the counter for the
// next forward.  So no consumer ever stalls on another CTA in the middle of its stream.
// `vals[i]` is the value of entry idx[i] = row_in_group * 16 + token (idx < 0: unused).
// T is float or int (integer sums are exact).  kRedBatch contributors are loaded per L2
// round trip in the reduction.
template <typename T, int NV, int kRedBatch = 8>
struct RowGroupFinisher {
  float* partials;     // the workspace's slots and counters, copied: taking the address of
  uint32_t* counters;  // a kernel parameter would move the parameter to local memory
  int cta;
  int rg[2];          // shared row groups: [0] the first of the range, [1] the last (-1: none)
  int first_cta[2];   // their first contributor
  int first_slot[2];  // and the slot that contributor stored into
  int ncontrib[2];    // number of contributors
  int pend;           // bit s: rg[s] has been staged

  __device__ __forceinline__ RowGroupFinisher(int64_t per_rg, int64_t units, int64_t grid, int64_t cta_,
                                              float* partials_, uint32_t* counters_)
      : partials(partials_), counters(counters_), cta((int)cta_), pend(0) {
    const int64_t u0 = split_start(cta_, units, grid), u1 = split_start(cta_ + 1, units, grid);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      rg[s] = -1;
      first_cta[s] = first_slot[s] = ncontrib[s] = 0;
      if (u1 <= u0) continue;
      const int64_t r = (s == 0 ? u0 : u1 - 1) / per_rg;
      if (s == 1 && r == u0 / per_rg) continue;
      const SplitInfo si = split_info(r, per_rg, units, grid);
      if (si.first_cta == si.last_cta) continue;
      rg[s] = (int)r;
      first_cta[s] = (int)si.first_cta;
      ncontrib[s] = (int)(si.last_cta - si.first_cta + 1);
      // only the first contributor can have the row group as its second one (slot side 1)
      first_slot[s] = (int)(si.first_cta * 2 + (split_start(si.first_cta, units, grid) < r * per_rg ? 1 : 0));
    }
  }

  template <typename Done>
  __device__ __forceinline__ void stage(int64_t r, const T (&vals)[NV], const int (&idx)[NV], Done done) {
    const int s = (r == rg[0]) ? 0 : (r == rg[1]) ? 1 : -1;
    if (s < 0) {
      done(r, vals);
      return;
    }
    T* slot = reinterpret_cast<T*>(partials) + (int64_t)(cta * 2 + s) * (kRowGroup * 16);
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (idx[i] >= 0) slot[idx[i]] = vals[i];
    pend |= 1 << s;
  }

  // Returns false if a bounded wait gave up.  `flags` is a 2-int shared array.
  //
  // Ordering: the consumer barrier orders every consumer's slot stores before thread 0's
  // arrival, which is an acq_rel atomic at GPU scope (release: this CTA's slots become
  // visible before the count; acquire, for the last arriver: the other contributors' slots
  // are visible to it), and the second barrier passes that on to the other consumers, which
  // read the slots from L2 (ld.cg).
  //
  // The last contributor reduces with all 128 consumer threads, both of its row groups at
  // once: work item j is the 16-byte quad (row, tokens 4i..4i+3) of one row group, and its
  // contributors' quads are loaded kRedBatch at a time and summed in CTA order.
  // `put(rg, entry, value)` stores one output.
  template <typename Put>
  __device__ __forceinline__ bool finish(int M, ConsumerSync& cs, int* flags, Put put) {
    if (pend == 0) return true;  // uniform: every consumer thread staged the same row groups
    if (!cs.sync()) return false;
    if (threadIdx.x == 0) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        int last = 0;
        if (pend & (1 << s)) {
          const unsigned old = atom_add_acq_rel_gpu(&counters[rg[s]], 1u);
          last = (old == (unsigned)(ncontrib[s] - 1)) ? 1 : 0;
        }
        flags[s] = last;
      }
    }
    if (!cs.sync()) return false;
    const int f0 = flags[0], f1 = flags[1];
    const int qm = (M + 3) >> 2, per = kRowGroup * qm;
    const T* base = reinterpret_cast<const T*>(partials);
    for (int w = threadIdx.x; w < (f0 + f1) * per; w += 128) {
      const int s = (f0 && w < per) ? 0 : 1;
      const int lin = w - ((f0 && s == 1) ? per : 0);
      const int e = (lin / qm) * 16 + (lin % qm) * 4;
      const int C = ncontrib[s], fc = first_cta[s], fs = first_slot[s];
      T acc[4] = {T(0), T(0), T(0), T(0)};
      for (int c0 = 0; c0 < C; c0 += kRedBatch) {
        T v[kRedBatch][4];
#pragma unroll
        for (int u = 0; u < kRedBatch; ++u) {
          const int c = c0 + u;
          if (c < C) {
            const int slot = (c == 0) ? fs : (fc + c) * 2;
            ldcg4(base + (int64_t)slot * (kRowGroup * 16) + e, v[u]);
          } else {
            v[u][0] = v[u][1] = v[u][2] = v[u][3] = T(0);
          }
        }
#pragma unroll
        for (int u = 0; u < kRedBatch; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[j] += v[u][j];
      }
      const int m0 = (lin % qm) * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (m0 + j < M) put((int64_t)rg[s], e + j, acc[j]);
    }
    if (threadIdx.x == 0) {
      if (f0) counters[rg[0]] = 0u;
      if (f1) counters[rg[1]] = 0u;
    }
    return true;
  }
};

// Completion for one token (M == 1) without atomics: the CTA that holds the first unit of a
// shared row group owns it -- it is the owner's last row group and every other contributor's
// first, so a CTA owns at most one.  Contributors store their 64 partial sums as 8-byte words
// (value bits, tag) into their slot of `tagged` and move on: no fence, no atomic, no wait.
// The owner keeps its own sums in shared memory and, at the end of its range, reads the
// contributors' words from L2 until every one carries the workspace's tag (an aligned 8-byte
// word is written and read as one access, so a word with the tag holds its value), adds them
// in CTA order (deterministic), writes the outputs and stores zero words back, so no slot
// holds a valid-looking word between forwards.  Owners wait only on higher-numbered CTAs,
// which never wait on lower ones, so the waits cannot form a cycle; every wait is bounded.
// Same interface as RowGroupFinisher; entries are idx = row_in_group * 16.
__device__ __forceinline__ void st_relaxed_b64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_b64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

template <int NV, int MAXM = 1>  // MAXM: 1 (M == 1) or 4 (M <= 4) tokens
struct OwnerFinisher {
  static constexpr int kSlotWords = kRowGroup * 4;  // words per slot (room for four tokens)
  static constexpr int PW = MAXM == 1 ? 1 : 2;      // words per work item
  uint64_t* tagged;  // [grid][2][kSlotWords] words (copied from the workspace, see RowGroupFinisher)
  int32_t* status;
  float* own;        // shared memory [64 * MAXM]: the owner's own partial sums
  uint32_t tag;
  int cta;
  int rg[2];         // shared row groups: [0] the first of the range, [1] the last (-1: none)
  int owned;         // side of the row group this CTA owns, -1 if none
  int others;        // contributors after this CTA to the owned row group
  int pend;          // 1 once the owned row group has been staged

  __device__ __forceinline__ OwnerFinisher(int64_t per_rg, int64_t units, int64_t grid, int64_t cta_,
                                           uint64_t* tagged_, uint32_t tag_, int32_t* status_, float* own_)
      : tagged(tagged_), status(status_), own(own_), tag(tag_), cta((int)cta_), owned(-1), others(0), pend(0) {
    const int64_t u0 = split_start(cta_, units, grid), u1 = split_start(cta_ + 1, units, grid);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      rg[s] = -1;
      if (u1 <= u0) continue;
      const int64_t r = (s == 0 ? u0 : u1 - 1) / per_rg;
      if (s == 1 && r == u0 / per_rg) continue;
      const SplitInfo si = split_info(r, per_rg, units, grid);
      if (si.first_cta == si.last_cta) continue;
      rg[s] = (int)r;
      if (si.first_cta == cta_) {
        owned = s;
        others = (int)(si.last_cta - si.first_cta);
      }
    }
  }

  // word of entry idx = row * 16 + token
  static __device__ __forceinline__ int word(int idx) { return (idx >> 4) * MAXM + (idx & 15); }
  __device__ __forceinline__ uint64_t* slot(int c, int side) const {
    return tagged + (int64_t)(c * 2 + side) * kSlotWords;
  }

  template <typename Done>
  __device__ __forceinline__ void stage(int64_t r, const float (&vals)[NV], const int (&idx)[NV], Done done) {
    const int s = (r == rg[0]) ? 0 : (r == rg[1]) ? 1 : -1;
    if (s < 0) {
      done(r, vals);
      return;
    }
    if (s == owned) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (idx[i] >= 0) own[word(idx[i])] = vals[i];
      pend = 1;
      return;
    }
    uint64_t* sl = slot(cta, s);
    const uint64_t hi = (uint64_t)tag << 32;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (idx[i] >= 0) st_relaxed_b64(sl + word(idx[i]), hi | __float_as_uint(vals[i]));
  }

  // Only the owner works here: work item j (thread j) is row j / (MAXM / PW), tokens
  // PW * (j % (MAXM / PW)) onward.  `put(rg, entry, value)` stores one output.
  template <typename Put>
  __device__ __forceinline__ bool finish(int M, ConsumerSync& cs, int* flags, Put put) {
    (void)flags;
    if (!pend) return true;  // uniform over the consumer threads
    if (!cs.sync()) return false;
    constexpr int IPR = MAXM / PW;  // items per row
    const int item = threadIdx.x;
    if (item >= kRowGroup * IPR) return true;
    const int row = item / IPR, m0 = (item % IPR) * PW;
    const int w0 = row * MAXM + m0;
    float acc[PW];
    bool need[PW];
#pragma unroll
    for (int j = 0; j < PW; ++j) {
      need[j] = m0 + j < M;
      acc[j] = own[w0 + j];
    }
    constexpr int B = 8;  // contributors loaded per L2 round trip
    for (int c0 = 0; c0 < others; c0 += B) {
      uint64_t v[B][PW];
#pragma unroll
      for (int u = 0; u < B; ++u)
        if (c0 + u < others)
#pragma unroll
          for (int j = 0; j < PW; ++j) v[u][j] = ld_relaxed_b64(slot(cta + 1 + c0 + u, 0) + w0 + j);
      // poll the whole batch: reload every word not yet tagged, one round trip per pass
      uint64_t t0 = 0;
      for (;;) {
        unsigned missing = 0;
#pragma unroll
        for (int u = 0; u < B; ++u)
#pragma unroll
          for (int j = 0; j < PW; ++j)
            if (c0 + u < others && need[j] && (uint32_t)(v[u][j] >> 32) != tag) missing |= 1u << u;
        if (!missing) break;
        if (t0 == 0) {
          t0 = global_ns();
        } else if (global_ns() - t0 > kWaitLimitNs) {
          atomicExch(status, kStatusTimeout);
          return false;
        }
#pragma unroll
        for (int u = 0; u < B; ++u)
          if (missing & (1u << u))
#pragma unroll
            for (int j = 0; j < PW; ++j) v[u][j] = ld_relaxed_b64(slot(cta + 1 + c0 + u, 0) + w0 + j);
      }
#pragma unroll
      for (int u = 0; u < B; ++u) {
        if (c0 + u >= others) continue;
#pragma unroll
        for (int j = 0; j < PW; ++j) {
          if (!need[j]) continue;
          acc[j] += __uint_as_float((uint32_t)v[u][j]);
          st_relaxed_b64(slot(cta + 1 + c0 + u, 0) + w0 + j, 0ull);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < PW; ++j)
      if (need[j]) put((int64_t)rg[owned], row * 16 + m0 + j, acc[j]);
    return true;
  }
};

}  // namespace qlin

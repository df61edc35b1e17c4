// Host side of libqlin: packers, device-image builders and the C ABI.
//
// Packers follow the three pages' methods (see include/qlin.h for the citations) with
// the readings the library documents: asymmetric round-to-nearest whose range always
// contains 0 with fp16 scales (GPTQ / SpQR pages), magnitude outlier selection and
// bi-level 3-bit statistics (SpQR page), the SmoothQuant smoothing fold with per-channel
// int8 weights (SmoothQuant page).  All arithmetic that decides a code is fp32 with IEEE
// division and round-half-to-even, compiled without fused multiply-add.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <limits>
#include <new>
#include <thread>
#include <vector>

#include "../../include/qlin.h"
#include "qlin_internal.h"

using namespace qlin;

// ------------------------------------------------------------------------------------
// fp16 helpers (round to nearest even)

static uint16_t f2h(float f) {
  uint32_t x;
  std::memcpy(&x, &f, 4);
  uint32_t sign = (x >> 16) & 0x8000u;
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);  // >= 65520 rounds to inf
  if (ax <= 0x33000000u) return (uint16_t)sign;              // <= 2^-25 rounds to 0
  uint32_t e = ax >> 23;
  if (e < 113) {  // fp16 subnormal
    uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126 - e;
    uint32_t r = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1u))) r++;
    return (uint16_t)(sign | r);
  }
  uint32_t r = ((e - 112) << 10) | ((ax >> 13) & 0x3FFu);
  uint32_t rem = ax & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) r++;
  return (uint16_t)(sign | r);
}

static float h2f(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1Fu;
  uint32_t m = h & 0x3FFu;
  uint32_t x;
  if (e == 0) {
    if (m == 0) {
      x = sign;
    } else {  // subnormal: value m * 2^-24
      float v = (float)m * 5.9604644775390625e-08f;
      std::memcpy(&x, &v, 4);
      x |= sign;
    }
  } else if (e == 31) {
    x = sign | 0x7F800000u | (m << 13);
  } else {
    x = sign | ((e + 112) << 23) | (m << 13);
  }
  float f;
  std::memcpy(&f, &x, 4);
  return f;
}

static inline bool is_finite_f(float v) { return std::isfinite(v); }

// ------------------------------------------------------------------------------------
// parallel-for over [0, n) in contiguous slices (deterministic: no cross-slice reduction)

static int host_threads() {
  unsigned n = std::thread::hardware_concurrency();
  if (n == 0) n = 1;
  return (int)std::min(n, 32u);
}

// fn(i) for i in [0, n), thread t of the pool taking i = t, t + T, t + 2T, ...: balances loops
// whose work grows with i (triangular matrices)
static void parallel_cyclic(int64_t n, const std::function<void(int64_t)>& fn) {
  const int nt = (int)std::min<int64_t>(host_threads(), std::max<int64_t>(n, 1));
  auto lane = [&](int t) {
    for (int64_t i = t; i < n; i += nt) fn(i);
  };
  std::vector<std::thread> th;
  for (int t = 1; t < nt; ++t) th.emplace_back(lane, t);
  lane(0);
  for (auto& x : th) x.join();
}

static void parallel_for(int64_t n, const std::function<void(int64_t, int64_t)>& fn) {
  int nt = host_threads();
  if (n < 64 || nt == 1) {
    fn(0, n);
    return;
  }
  nt = (int)std::min<int64_t>(nt, n);
  std::vector<std::thread> th;
  int64_t chunk = (n + nt - 1) / nt;
  for (int t = 1; t < nt; ++t) {
    int64_t b = t * chunk, e = std::min<int64_t>(n, b + chunk);
    if (b >= e) break;
    th.emplace_back(fn, b, e);
  }
  fn(0, std::min<int64_t>(n, chunk));
  for (auto& x : th) x.join();
}

// ------------------------------------------------------------------------------------
// Q_b: asymmetric round-to-nearest over one group, range always containing 0.
//   lo = min(0, min v), hi = max(0, max v); hi == lo -> scale 1, zero 0;
//   scale = fp16((hi - lo) / (2^b - 1)), 2^-24 if that is 0; z = clamp(rint(-lo/scale));
//   q = clamp(rint(v/scale) + z).  `valid` restricts the min/max (SpQR first level).

struct RtnStats {
  uint16_t scale_h;
  float scale;
  float zero;
  bool overflow;
};

static RtnStats rtn_stats(const float* v, const uint8_t* valid, int n, int bits) {
  const float qmax = (float)((1 << bits) - 1);
  float vmin = 0.f, vmax = 0.f;
  bool any = false;
  for (int i = 0; i < n; ++i) {
    if (valid && !valid[i]) continue;
    if (!any) {
      vmin = vmax = v[i];
      any = true;
    } else {
      vmin = std::min(vmin, v[i]);
      vmax = std::max(vmax, v[i]);
    }
  }
  float lo = std::min(0.f, vmin);
  float hi = std::max(0.f, vmax);
  RtnStats r{};
  if (hi == lo) {
    r.scale_h = 0x3C00;  // 1.0
    r.scale = 1.f;
    r.zero = 0.f;
    return r;
  }
  float s32 = (hi - lo) / qmax;
  uint16_t h = f2h(s32);
  if ((h & 0x7C00u) == 0x7C00u) {
    r.overflow = true;
    return r;
  }
  if ((h & 0x7FFFu) == 0) h = 0x0001;  // 2^-24
  r.scale_h = h;
  r.scale = h2f(h);
  float z = std::nearbyint(-lo / r.scale);
  z = std::min(std::max(z, 0.f), qmax);
  r.zero = z + 0.0f;  // -0 -> +0
  return r;
}

static inline int rtn_code(float v, const RtnStats& st, int bits) {
  const float qmax = (float)((1 << bits) - 1);
  float q = std::nearbyint(v / st.scale) + st.zero;
  q = std::min(std::max(q, 0.f), qmax);
  return (int)q;
}

// ------------------------------------------------------------------------------------
// the layer handle

// qlin_forward_host's captured steps (H2D copy, forward, D2H copy), one per set of pointers
struct HostGraph {
  const void* xh;
  void* yh;
  void* xd;
  void* yd;
  const uint8_t* dev;
  int M;
  cudaStream_t stream;
  cudaGraphExec_t exec;
  uint64_t used;
};

struct qlin_layer {
  ~qlin_layer() {
    for (auto& g : host_graphs) cudaGraphExecDestroy(g.exec);  // errors at process exit are moot
  }
  std::vector<HostGraph> host_graphs;
  uint64_t host_graph_clock = 0;
  int format = 0;
  int N = 0, K = 0;
  float alpha = 0.f, frac = 0.f;
  int64_t nnz = 0;
  // canonical arrays
  std::vector<uint32_t> codes;
  std::vector<uint16_t> scale, zero;
  std::vector<int32_t> perm;  // W4 act-order: permuted column j is input channel perm[j] (empty: none)
  std::vector<uint8_t> codes3, qs3, qz3;
  std::vector<uint16_t> stats;
  std::vector<int32_t> rowptr;
  std::vector<int16_t> col;
  std::vector<uint16_t> val;
  std::vector<int8_t> qw;
  std::vector<float> sw, s, s_inv;
  // device image and its sections
  std::vector<uint8_t> image;
  size_t sec_units = 0, sec_offs = 0, sec_ents = 0, sec_sw = 0, sec_sinv = 0, sec_perm = 0, sec_w2 = 0;
  int RG = 0, KU = 0;  // row groups, K units per row group
  // bound state
  uint8_t* dev = nullptr;
  size_t dev_bytes = 0;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  int ws_maxM = 0;
  Workspace wsv{};
  int grid = 0;
};

// SM count of the current device, looked up once per device
static int sm_count_cached() {
  static std::atomic<int> cached[64];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  if (dev >= 0 && dev < 64 && (n = cached[dev].load()) > 0) return n;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 152;
  }
  if (dev >= 0 && dev < 64) cached[dev].store(n);
  return n;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ------------------------------------------------------------------------------------
// W4 g128

static void build_w4_image(qlin_layer* L, const std::vector<uint8_t>& q);

static qlin_status build_w4(qlin_layer* L, const float* W) {
  const int N = L->N, K = L->K, G = K / kW4Group;
  L->scale.assign((size_t)N * G, 0);
  L->zero.assign((size_t)N * G, 0);
  std::vector<uint8_t> q((size_t)N * K);
  std::atomic<bool> bad{false};
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n) {
      const float* row = W + (size_t)n * K;
      for (int g = 0; g < G; ++g) {
        RtnStats st = rtn_stats(row + g * kW4Group, nullptr, kW4Group, 4);
        if (st.overflow) {
          bad = true;
          return;
        }
        L->scale[(size_t)n * G + g] = st.scale_h;
        L->zero[(size_t)n * G + g] = f2h(st.zero);
        for (int i = 0; i < kW4Group; ++i)
          q[(size_t)n * K + g * kW4Group + i] = (uint8_t)rtn_code(row[g * kW4Group + i], st, 4);
      }
    }
  });
  if (bad) return QLIN_ERR_INVALID_ARG;
  build_w4_image(L, q);
  return QLIN_OK;
}

// Canonical codes [N][K/8] and the device image from codes q [N][K] (scale and zero set).
static void build_w4_image(qlin_layer* L, const std::vector<uint8_t>& q) {
  const int N = L->N, K = L->K, G = K / kW4Group;
  L->codes.assign((size_t)N * (K / 8), 0u);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n)
      for (int j = 0; j < K / 8; ++j) {
        uint32_t w = 0;
        for (int i = 0; i < 8; ++i) w |= (uint32_t)q[(size_t)n * K + 8 * j + i] << (4 * i);
        L->codes[(size_t)n * (K / 8) + j] = w;
      }
  });

  // device image: units [RG][G], codes in A-fragment order + (scale, zero) per row
  const int RG = (N + kRowGroup - 1) / kRowGroup;
  L->RG = RG;
  L->KU = G;
  L->sec_units = 0;
  const size_t units_bytes = align256((size_t)RG * G * kW4UnitBytes);
  L->sec_perm = units_bytes;
  L->image.assign(units_bytes + (L->perm.empty() ? 0 : align256((size_t)K * 4)), 0);
  uint8_t* img = L->image.data();
  if (!L->perm.empty()) std::memcpy(img + L->sec_perm, L->perm.data(), (size_t)K * 4);
  parallel_for(RG, [&](int64_t b, int64_t e) {
    for (int64_t rg = b; rg < e; ++rg) {
      for (int g = 0; g < G; ++g) {
        uint8_t* unit = img + ((size_t)rg * G + g) * kW4UnitBytes;
        uint32_t* cw = reinterpret_cast<uint32_t*>(unit);
        uint16_t* st = reinterpret_cast<uint16_t*>(unit + kW4CodeBytes);
        for (int rt = 0; rt < 4; ++rt) {
          for (int kb = 0; kb < 2; ++kb) {
            for (int lane = 0; lane < 32; ++lane) {
              const int gg = lane >> 2, t = lane & 3;
              for (int j = 0; j < 4; ++j) {
                const int k0 = g * kW4Group + kb * 64 + 16 * j;
                auto code = [&](int r, int k) -> uint32_t {
                  int64_t n = rg * kRowGroup + rt * 16 + r;
                  return n < N ? q[(size_t)n * K + k] : 0u;
                };
                uint32_t w = 0;
                w |= code(gg, k0 + 2 * t) << 0;
                w |= code(gg + 8, k0 + 2 * t) << 4;
                w |= code(gg, k0 + 2 * t + 8) << 8;
                w |= code(gg + 8, k0 + 2 * t + 8) << 12;
                w |= code(gg, k0 + 2 * t + 1) << 16;
                w |= code(gg + 8, k0 + 2 * t + 1) << 20;
                w |= code(gg, k0 + 2 * t + 9) << 24;
                w |= code(gg + 8, k0 + 2 * t + 9) << 28;
                cw[((rt * 2 + kb) * 32 + lane) * 4 + j] = w;
              }
            }
          }
          for (int r = 0; r < 16; ++r) {
            int64_t n = rg * kRowGroup + rt * 16 + r;
            st[(rt * 16 + r) * 2 + 0] = n < N ? L->scale[(size_t)n * G + g] : 0;
            st[(rt * 16 + r) * 2 + 1] = n < N ? L->zero[(size_t)n * G + g] : 0;
          }
        }
      }
    }
  });
}

// ------------------------------------------------------------------------------------
// GPTQ W4 g128 (GPTQ page, "Makale Bülteni — GPTQ" intro and "İddia ve Gerçeklik: GPTQ"):
// the inverse Hessian comes from the covariance of the layer inputs and is stabilised by a
// Cholesky decomposition; columns are quantized in order and each column's rounding error is
// spread at once over the columns not yet quantized.  The steps the page leaves open are read
// as: H = Xcal^T Xcal (fp64); an always-zero input column gets H_kk = 1 and zero weights;
// H += damp * mean(diag H) * I; U = the upper Cholesky factor of H^-1 (H^-1 = U^T U); at the
// first column of each 128-group the group's scale and zero are the round-to-nearest ones of
// the group's current weights (as fp32); a column's code is the round-to-nearest code with
// them, and with e = (w_k - w_hat_k) / U_kk every later weight of the row becomes
// w_j - e * U_kj (fp64).  The page batches the updates of a 128-block for speed on a GPU; on
// the host each row is independent and is updated column by column (the same arithmetic).

static constexpr int kGptqMaxK = 8192;  // H and its factors are K x K fp64 on the host

// sum of a[p] * b[p], p < n, in four interleaved partial sums
static inline double dot4(const double* a, const double* b, int64_t n) {
  double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
  int64_t p = 0;
  for (; p + 4 <= n; p += 4) {
    s0 += a[p] * b[p];
    s1 += a[p + 1] * b[p + 1];
    s2 += a[p + 2] * b[p + 2];
    s3 += a[p + 3] * b[p + 3];
  }
  for (; p < n; ++p) s0 += a[p] * b[p];
  return (s0 + s1) + (s2 + s3);
}

// U with H^-1 = U^T U, U upper triangular with a positive diagonal: with J the order reversal,
// J H J = L L^T (lower Cholesky factor L) gives H = V V^T for the upper V = J L J, and
// H^-1 = (V^-1)^T V^-1, so U = V^-1.  H is overwritten.  Returns false if H is not positive
// definite.
static bool gptq_inverse_factor(std::vector<double>& H, int K, std::vector<double>& U) {
  // L (lower, row-major) of A = J H J, computed in place over A
  std::vector<double> A((size_t)K * K);
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < K; ++j) A[(size_t)i * K + j] = H[(size_t)(K - 1 - i) * K + (K - 1 - j)];
  std::vector<double>().swap(H);
  // right-looking blocked Cholesky, panels of kB columns: factor the diagonal block, solve the
  // rows below it, then subtract the panel's contribution from the trailing lower triangle
  constexpr int kB = 64;
  std::atomic<bool> not_pd{false};
  for (int jb = 0; jb < K; jb += kB) {
    const int je = std::min(K, jb + kB);
    for (int j = jb; j < je; ++j) {  // diagonal block (columns of earlier panels already applied)
      double* Lj = &A[(size_t)j * K];
      double d = Lj[j];
      for (int p = jb; p < j; ++p) d -= Lj[p] * Lj[p];
      if (!(d > 0.0)) return false;
      Lj[j] = std::sqrt(d);
      for (int i = j + 1; i < je; ++i) {
        double* Li = &A[(size_t)i * K];
        double v = Li[j];
        for (int p = jb; p < j; ++p) v -= Li[p] * Lj[p];
        Li[j] = v / Lj[j];
      }
    }
    const int64_t rest = K - je;
    if (rest <= 0) break;
    auto panel = [&](int64_t b, int64_t e) {  // rows below the block: L[i][jb..je)
      for (int64_t r = b; r < e; ++r) {
        double* Li = &A[(size_t)(je + r) * K];
        for (int j = jb; j < je; ++j) {
          const double* Lj = &A[(size_t)j * K];
          Li[j] = (Li[j] - dot4(Li + jb, Lj + jb, j - jb)) / Lj[j];
        }
      }
    };
    auto trailing = [&](int64_t r) {  // row je + r: A[i][j] -= sum over the panel, je <= j <= i
      const int64_t i = je + r;
      double* Ai = &A[(size_t)i * K];
      for (int64_t j = je; j <= i; ++j) Ai[j] -= dot4(Ai + jb, &A[(size_t)j * K + jb], je - jb);
    };
    if (rest * (je - jb) > (1 << 14)) parallel_for(rest, panel); else panel(0, rest);
    if (rest * rest > (1 << 14)) {
      parallel_cyclic(rest, trailing);
    } else {
      for (int64_t r = 0; r < rest; ++r) trailing(r);
    }
  }
  (void)not_pd;
  // V = J L J (upper): V[i][j] = L[K-1-i][K-1-j]; U = V^-1 column by column (back substitution),
  // column j of U kept as row j of UT so both operands are contiguous
  auto V = [&](int i, int j) { return A[(size_t)(K - 1 - i) * K + (K - 1 - j)]; };
  std::vector<double> Vr((size_t)K * K, 0.0);  // V row-major, upper part
  for (int i = 0; i < K; ++i)
    for (int j = i; j < K; ++j) Vr[(size_t)i * K + j] = V(i, j);
  std::vector<double>().swap(A);
  std::vector<double> UT((size_t)K * K, 0.0);
  parallel_cyclic(K, [&](int64_t j) {  // column j costs ~j^2: cyclic assignment balances them
    double* u = &UT[(size_t)j * K];
    for (int64_t i = j; i >= 0; --i) {
      const double* Vi = &Vr[(size_t)i * K];
      const double v = ((i == j) ? 1.0 : 0.0) - dot4(Vi + i + 1, u + i + 1, j - i);
      u[i] = v / Vi[i];
    }
  });
  U.assign((size_t)K * K, 0.0);
  for (int j = 0; j < K; ++j)
    for (int i = 0; i <= j; ++i) U[(size_t)i * K + j] = UT[(size_t)j * K + i];
  return true;
}

static qlin_status build_w4_gptq(qlin_layer* L, const float* W, const float* Xcal, int S, double damp,
                                 bool act_order) {
  const int N = L->N, K = L->K, G = K / kW4Group;
  // H = Xcal^T Xcal over the calibration rows, in row order
  std::vector<double> H((size_t)K * K, 0.0);
  parallel_for(K, [&](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i)
      for (int s = 0; s < S; ++s) {
        const float* x = Xcal + (size_t)s * K;
        const double xi = (double)x[i];
        if (xi == 0.0) continue;
        double* Hi = &H[(size_t)i * K];
        for (int j = 0; j < K; ++j) Hi[j] += xi * (double)x[j];
      }
  });
  // act-order (GPTQ page, "İddia ve Gerçeklik: GPTQ", last paragraph): columns by decreasing
  // diag(H) (an always-zero input counted as 1), ties to the smaller index; the permuted layer
  // W[:, perm] is quantized under H[perm][perm], so its 128-groups are contiguous in that order
  std::vector<float> Wp;
  if (act_order) {
    std::vector<double> d(K);
    for (int k = 0; k < K; ++k) d[k] = H[(size_t)k * K + k] == 0.0 ? 1.0 : H[(size_t)k * K + k];
    L->perm.resize(K);
    for (int k = 0; k < K; ++k) L->perm[k] = k;
    std::stable_sort(L->perm.begin(), L->perm.end(), [&](int32_t a, int32_t b) { return d[a] > d[b]; });
    std::vector<double> Hp((size_t)K * K);
    parallel_for(K, [&](int64_t b, int64_t e) {
      for (int64_t i = b; i < e; ++i)
        for (int j = 0; j < K; ++j) Hp[(size_t)i * K + j] = H[(size_t)L->perm[i] * K + L->perm[j]];
    });
    H.swap(Hp);
    Wp.resize((size_t)N * K);
    parallel_for(N, [&](int64_t b, int64_t e) {
      for (int64_t n = b; n < e; ++n)
        for (int j = 0; j < K; ++j) Wp[(size_t)n * K + j] = W[(size_t)n * K + L->perm[j]];
    });
    W = Wp.data();
  }
  std::vector<uint8_t> dead(K, 0);
  double diag = 0.0;
  for (int k = 0; k < K; ++k) {
    if (H[(size_t)k * K + k] == 0.0) {
      dead[k] = 1;
      H[(size_t)k * K + k] = 1.0;
    }
    diag += H[(size_t)k * K + k];
  }
  const double add = damp * (diag / K);
  for (int k = 0; k < K; ++k) H[(size_t)k * K + k] += add;
  std::vector<double> U;
  if (!gptq_inverse_factor(H, K, U)) return QLIN_ERR_INVALID_ARG;

  L->scale.assign((size_t)N * G, 0);
  L->zero.assign((size_t)N * G, 0);
  std::vector<uint8_t> q((size_t)N * K);
  std::atomic<bool> bad{false};
  // Rows are independent: they are taken kGptqTile at a time, transposed to [K][tile], so each
  // element of U read from memory serves the whole tile and the update runs along contiguous
  // rows.  Every weight still receives its updates one by one in column order, as products
  // then differences (the oracle's arithmetic, bit for bit).
  constexpr int kGptqTile = 32;
  const int64_t tiles = (N + kGptqTile - 1) / kGptqTile;
  parallel_for(tiles, [&](int64_t tb, int64_t tend) {
    std::vector<double> wt((size_t)K * kGptqTile);
    std::vector<float> gv(kW4Group);
    RtnStats st[kGptqTile];
    double ek[kGptqTile];
    for (int64_t tile = tb; tile < tend && !bad; ++tile) {
      const int64_t n0 = tile * kGptqTile;
      const int nr = (int)std::min<int64_t>(kGptqTile, N - n0);
      for (int k = 0; k < K; ++k)
        for (int r = 0; r < nr; ++r) wt[(size_t)k * kGptqTile + r] = dead[k] ? 0.0 : (double)W[(size_t)(n0 + r) * K + k];
      for (int k = 0; k < K; ++k) {
        const int g = k / kW4Group;
        if (k % kW4Group == 0) {
          for (int r = 0; r < nr; ++r) {
            for (int i = 0; i < kW4Group; ++i) gv[i] = (float)wt[(size_t)(k + i) * kGptqTile + r];
            st[r] = rtn_stats(gv.data(), nullptr, kW4Group, 4);
            if (st[r].overflow) {
              bad = true;
              return;
            }
            L->scale[(size_t)(n0 + r) * G + g] = st[r].scale_h;
            L->zero[(size_t)(n0 + r) * G + g] = f2h(st[r].zero);
          }
        }
        const double ukk = U[(size_t)k * K + k];
        for (int r = 0; r < nr; ++r) {
          const double wk = wt[(size_t)k * kGptqTile + r];
          const int code = rtn_code((float)wk, st[r], 4);
          q[(size_t)(n0 + r) * K + k] = (uint8_t)code;
          const float w_hat = ((float)code - st[r].zero) * st[r].scale;
          ek[r] = (wk - (double)w_hat) / ukk;
        }
        const double* Uk = &U[(size_t)k * K];
        for (int j = k + 1; j < K; ++j) {
          const double u = Uk[j];
          double* wj = &wt[(size_t)j * kGptqTile];
          for (int r = 0; r < nr; ++r) wj[r] -= ek[r] * u;
        }
      }
    }
  });
  if (bad) return QLIN_ERR_INVALID_ARG;
  build_w4_image(L, q);
  return QLIN_OK;
}

// ------------------------------------------------------------------------------------
// SpQR

// Outlier mask: the nnz largest |w|, ties broken toward the smaller linear index.
// Radix select on the magnitude bit pattern (monotone in |w| for finite values).
static void spqr_outliers(const float* W, int64_t total, int64_t nnz, int N, int K,
                          std::vector<uint8_t>& mask) {
  mask.assign((size_t)total, 0);
  if (nnz <= 0) return;
  auto mag = [&](int64_t i) {
    uint32_t u;
    std::memcpy(&u, W + i, 4);
    return u & 0x7FFFFFFFu;
  };
  int nt = host_threads();
  // pass 1: high 16 bits
  std::vector<std::vector<int64_t>> hist(nt, std::vector<int64_t>(1 << 16, 0));
  {
    std::vector<std::thread> th;
    int64_t chunk = (total + nt - 1) / nt;
    for (int t = 0; t < nt; ++t)
      th.emplace_back([&, t]() {
        int64_t b = t * chunk, e = std::min(total, b + chunk);
        for (int64_t i = b; i < e; ++i) hist[t][mag(i) >> 16]++;
      });
    for (auto& x : th) x.join();
  }
  std::vector<int64_t> h(1 << 16, 0);
  for (int t = 0; t < nt; ++t)
    for (int i = 0; i < (1 << 16); ++i) h[i] += hist[t][i];
  int64_t above = 0;
  int hb = (1 << 16) - 1;
  for (; hb >= 0; --hb) {
    if (above + h[hb] >= nnz) break;
    above += h[hb];
  }
  // pass 2: low 16 bits within bucket hb
  for (int t = 0; t < nt; ++t) std::fill(hist[t].begin(), hist[t].end(), 0);
  {
    std::vector<std::thread> th;
    int64_t chunk = (total + nt - 1) / nt;
    for (int t = 0; t < nt; ++t)
      th.emplace_back([&, t]() {
        int64_t b = t * chunk, e = std::min(total, b + chunk);
        for (int64_t i = b; i < e; ++i) {
          uint32_t m = mag(i);
          if ((int)(m >> 16) == hb) hist[t][m & 0xFFFFu]++;
        }
      });
    for (auto& x : th) x.join();
  }
  std::fill(h.begin(), h.end(), 0);
  for (int t = 0; t < nt; ++t)
    for (int i = 0; i < (1 << 16); ++i) h[i] += hist[t][i];
  int lb = (1 << 16) - 1;
  for (; lb >= 0; --lb) {
    if (above + h[lb] >= nnz) break;
    above += h[lb];
  }
  const uint32_t T = ((uint32_t)hb << 16) | (uint32_t)lb;
  const int64_t need_ties = nnz - above;  // entries equal to T to take, in index order
  // per-row tie counts -> quota per row
  std::vector<int64_t> ties(N, 0);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n) {
      int64_t c = 0;
      for (int k = 0; k < K; ++k) c += mag(n * K + k) == T;
      ties[n] = c;
    }
  });
  std::vector<int64_t> quota(N, 0);
  int64_t left = need_ties;
  for (int n = 0; n < N; ++n) {
    quota[n] = std::min(left, ties[n]);
    left -= quota[n];
  }
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n) {
      int64_t qn = quota[n];
      for (int k = 0; k < K; ++k) {
        uint32_t m = mag(n * K + k);
        if (m > T) {
          mask[(size_t)n * K + k] = 1;
        } else if (m == T && qn > 0) {
          mask[(size_t)n * K + k] = 1;
          --qn;
        }
      }
    }
  });
}

static void put_bits3(std::vector<uint8_t>& stream, size_t row_off, int idx, int code) {
  size_t bit = (size_t)3 * idx;
  for (int b = 0; b < 3; ++b, ++bit)
    if ((code >> b) & 1) stream[row_off + bit / 8] |= (uint8_t)(1u << (bit % 8));
}

static void build_spqr_image(qlin_layer* L, const std::vector<uint8_t>& q, const std::vector<uint8_t>& qs,
                             const std::vector<uint8_t>& qz);

static qlin_status build_spqr(qlin_layer* L, const float* W) {
  const int N = L->N, K = L->K;
  const int G = K / 16, S = K / kSpqrSuper;
  const int64_t total = (int64_t)N * K;
  const int64_t nnz = (int64_t)std::floor((double)L->frac * (double)total);
  L->nnz = nnz;
  std::vector<uint8_t> mask;
  spqr_outliers(W, total, nnz, N, K, mask);

  std::vector<uint8_t> q((size_t)total);
  std::vector<float> D((size_t)total);
  std::vector<uint8_t> qs((size_t)N * G), qz((size_t)N * G);
  L->stats.assign((size_t)N * S * 4, 0);
  std::atomic<bool> bad{false};
  parallel_for(N, [&](int64_t b, int64_t e) {
    std::vector<float> sg(G), zg(G);
    for (int64_t n = b; n < e && !bad; ++n) {
      const float* row = W + (size_t)n * K;
      const uint8_t* mrow = mask.data() + (size_t)n * K;
      // first level over the non-outliers of each 16-group
      for (int g = 0; g < G; ++g) {
        uint8_t valid[16];
        for (int i = 0; i < 16; ++i) valid[i] = !mrow[g * 16 + i];
        RtnStats st = rtn_stats(row + g * 16, valid, 16, 3);
        if (st.overflow) {
          bad = true;
          return;
        }
        sg[g] = st.scale;
        zg[g] = st.zero;
      }
      // second level per supergroup, then the dense codes
      for (int s = 0; s < S; ++s) {
        RtnStats a = rtn_stats(&sg[s * 16], nullptr, 16, 3);
        RtnStats c = rtn_stats(&zg[s * 16], nullptr, 16, 3);
        if (a.overflow || c.overflow) {
          bad = true;
          return;
        }
        uint16_t* st = &L->stats[((size_t)n * S + s) * 4];
        st[0] = a.scale_h;
        st[1] = f2h(a.zero);
        st[2] = c.scale_h;
        st[3] = f2h(c.zero);
        for (int gg = 0; gg < 16; ++gg) {
          const int g = s * 16 + gg;
          const int cqs = rtn_code(sg[g], a, 3);
          const int cqz = rtn_code(zg[g], c, 3);
          qs[(size_t)n * G + g] = (uint8_t)cqs;
          qz[(size_t)n * G + g] = (uint8_t)cqz;
          const float sh = ((float)cqs - a.zero) * a.scale;
          const float zh = ((float)cqz - c.zero) * c.scale;
          for (int i = 0; i < 16; ++i) {
            const int k = g * 16 + i;
            int code = 0;
            if (sh != 0.f) {
              float t = std::nearbyint(row[k] / sh + zh);
              t = std::min(std::max(t, 0.f), 7.f);
              code = (int)t;
            }
            q[(size_t)n * K + k] = (uint8_t)code;
            D[(size_t)n * K + k] = ((float)code - zh) * sh;
          }
        }
      }
    }
  });
  if (bad) return QLIN_ERR_INVALID_ARG;

  // canonical streams and CSR
  const size_t cb = (size_t)3 * K / 8, sb = (size_t)3 * G / 8;
  L->codes3.assign((size_t)N * cb, 0);
  L->qs3.assign((size_t)N * sb, 0);
  L->qz3.assign((size_t)N * sb, 0);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n) {
      for (int k = 0; k < K; ++k) put_bits3(L->codes3, n * cb, k, q[(size_t)n * K + k]);
      for (int g = 0; g < G; ++g) {
        put_bits3(L->qs3, n * sb, g, qs[(size_t)n * G + g]);
        put_bits3(L->qz3, n * sb, g, qz[(size_t)n * G + g]);
      }
    }
  });
  L->rowptr.assign(N + 1, 0);
  for (int n = 0; n < N; ++n) {
    int c = 0;
    const uint8_t* mrow = mask.data() + (size_t)n * K;
    for (int k = 0; k < K; ++k) c += mrow[k];
    L->rowptr[n + 1] = L->rowptr[n] + c;
  }
  L->col.assign((size_t)nnz, 0);
  L->val.assign((size_t)nnz, 0);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e && !bad; ++n) {
      int64_t p = L->rowptr[n];
      for (int k = 0; k < K; ++k) {
        if (!mask[(size_t)n * K + k]) continue;
        float r = W[(size_t)n * K + k] - D[(size_t)n * K + k];
        uint16_t h = f2h(r);
        if ((h & 0x7C00u) == 0x7C00u) {
          bad = true;
          return;
        }
        L->col[p] = (int16_t)k;
        L->val[p] = h;
        ++p;
      }
    }
  });
  if (bad) return QLIN_ERR_INVALID_ARG;
  build_spqr_image(L, q, qs, qz);
  return QLIN_OK;
}

// Device image from the codes q [N][K], qs, qz [N][K/16] and the handle's stats and CSR.
static void build_spqr_image(qlin_layer* L, const std::vector<uint8_t>& q, const std::vector<uint8_t>& qs,
                             const std::vector<uint8_t>& qz) {
  const int N = L->N, K = L->K;
  const int G = K / 16, S = K / kSpqrSuper;
  const int64_t nnz = L->nnz;
  const int RG = (N + kRowGroup - 1) / kRowGroup;
  L->RG = RG;
  L->KU = S;
  const size_t units = (size_t)RG * S;
  const size_t units_bytes = align256(units * kSpqrUnitBytes);
  const size_t offs_bytes = align256((units * 4 + 1) * 4);
  const size_t ents_bytes = align256((size_t)std::max<int64_t>(nnz, 1) * 4);
  L->sec_units = 0;
  L->sec_offs = units_bytes;
  L->sec_ents = units_bytes + offs_bytes;
  L->image.assign(units_bytes + offs_bytes + ents_bytes, 0);
  uint8_t* img = L->image.data();
  auto codeat = [&](int64_t n, int k) -> uint32_t { return n < N ? q[(size_t)n * K + k] : 0u; };
  auto qsat = [&](int64_t n, int g) -> uint32_t { return n < N ? qs[(size_t)n * G + g] : 0u; };
  auto qzat = [&](int64_t n, int g) -> uint32_t { return n < N ? qz[(size_t)n * G + g] : 0u; };
  parallel_for(RG, [&](int64_t b, int64_t e) {
    for (int64_t rg = b; rg < e; ++rg) {
      for (int s = 0; s < S; ++s) {
        uint8_t* unit = img + (rg * S + s) * kSpqrUnitBytes;
        uint32_t* cw = reinterpret_cast<uint32_t*>(unit);
        uint8_t* qq = unit + kSpqrCodeBytes;
        uint16_t* st = reinterpret_cast<uint16_t*>(unit + kSpqrCodeBytes + kSpqrQsqzBytes);
        for (int rt = 0; rt < 4; ++rt) {
          const int64_t r0 = rg * kRowGroup + rt * 16;
          for (int blk = 0; blk < 2; ++blk) {
            const int kb0 = s * kSpqrSuper + blk * 128;  // first k of the block
            uint32_t* words = cw + (size_t)(rt * 2 + blk) * 32 * 6;
            uint8_t* qsqz = qq + (size_t)(rt * 2 + blk) * 96;
            for (int lane = 0; lane < 32; ++lane) {
              const int gq = lane >> 2, t = lane & 3;
              uint32_t w[6] = {0, 0, 0, 0, 0, 0};
              // A register r -> (row, group in block)
              auto rowof = [&](int r) { return r0 + gq + ((r & 1) ? 8 : 0); };
              auto grpof = [&](int r) { return t + ((r & 2) ? 4 : 0); };
              for (int j = 0; j < 8; ++j) {
                for (int r = 0; r < 4; ++r) {
                  const int64_t n = rowof(r);
                  const int k_lo = kb0 + 16 * grpof(r) + 2 * j;
                  const uint32_t lo = codeat(n, k_lo), hi = codeat(n, k_lo + 1);
                  if (j <= 4) {
                    const int i = 4 * j + r;
                    if (i < 18) {
                      const int wi = i / 3, f = (i % 3) * 2;  // fields 0, 2, 4
                      w[wi] |= lo << (3 * f);
                      w[wi] |= hi << (16 + 3 * f);
                    } else {
                      const int base = 3 * (i - 18);
                      for (int bb = 0; bb < 3; ++bb) {
                        w[base + bb] |= ((lo >> bb) & 1u) << 15;
                        w[base + bb] |= ((hi >> bb) & 1u) << 31;
                      }
                    }
                  } else {
                    const int i = 4 * (j - 5) + r;
                    const int wi = i / 2, f = (i % 2) * 2 + 1;  // fields 1, 3
                    w[wi] |= lo << (3 * f);
                    w[wi] |= hi << (16 + 3 * f);
                  }
                }
              }
              for (int x = 0; x < 6; ++x) words[lane * 6 + x] = w[x];
              // 24-bit (qs, qz) field of the accumulator-side pairs
              uint32_t f24 = 0;
              for (int i = 0; i < 4; ++i) {
                const int64_t n = r0 + gq + ((i & 2) ? 8 : 0);
                const int gg = s * 16 + blk * 8 + 2 * t + (i & 1);
                f24 |= qsat(n, gg) << (6 * i);
                f24 |= qzat(n, gg) << (6 * i + 3);
              }
              for (int bb = 0; bb < 24; ++bb) {
                const int bit = 24 * lane + bb;
                if ((f24 >> bb) & 1u) qsqz[bit / 8] |= (uint8_t)(1u << (bit % 8));
              }
            }
          }
          for (int r = 0; r < 16; ++r) {
            const int64_t n = r0 + r;
            for (int x = 0; x < 4; ++x)
              st[(rt * 16 + r) * 4 + x] = n < N ? L->stats[((size_t)n * S + s) * 4 + x] : 0;
          }
        }
      }
    }
  });
  // outlier buckets [unit][rt], entries (val << 16 | k in unit << 4 | row in tile)
  uint32_t* offs = reinterpret_cast<uint32_t*>(img + L->sec_offs);
  uint32_t* ents = reinterpret_cast<uint32_t*>(img + L->sec_ents);
  {
    std::vector<uint32_t> cnt(units * 4, 0);
    for (int n = 0; n < N; ++n) {
      const int rg = n / kRowGroup, rt = (n % kRowGroup) / 16;
      for (int p = L->rowptr[n]; p < L->rowptr[n + 1]; ++p) {
        const int s = L->col[p] / kSpqrSuper;
        cnt[((size_t)rg * S + s) * 4 + rt]++;
      }
    }
    uint32_t acc = 0;
    for (size_t i = 0; i < units * 4; ++i) {
      offs[i] = acc;
      acc += cnt[i];
    }
    offs[units * 4] = acc;
    std::vector<uint32_t> fill(offs, offs + units * 4);
    for (int n = 0; n < N; ++n) {
      const int rg = n / kRowGroup, rt = (n % kRowGroup) / 16, rr = n % 16;
      for (int p = L->rowptr[n]; p < L->rowptr[n + 1]; ++p) {
        const int k = L->col[p];
        const int s = k / kSpqrSuper;
        const size_t bkt = ((size_t)rg * S + s) * 4 + rt;
        ents[fill[bkt]++] = ((uint32_t)L->val[p] << 16) | ((uint32_t)(k % kSpqrSuper) << 4) | (uint32_t)rr;
      }
    }
    // Order inside a bucket: by quad (row & 7), then row, then k -- an MMA lane quad g owns
    // the accumulators of rows g and g + 8, so each quad's outliers are one run, and so is
    // each row's.  With at least 8 entries, bits 12..15 of entries 0..7 hold the entry counts
    // of quads 0..7 (15 in all eight when some quad has 15 or more).
    auto key = [](uint32_t e) {
      const uint32_t r = e & 15u;
      return (((r & 7u) << 1 | (r >> 3)) << 8) | ((e >> 4) & 255u);
    };
    for (size_t b = 0; b < units * 4; ++b) {
      uint32_t* e0 = ents + offs[b];
      const uint32_t n = offs[b + 1] - offs[b];
      std::sort(e0, e0 + n, [&](uint32_t a, uint32_t c) { return key(a) < key(c); });
      if (n < 8) continue;
      uint32_t cnt[8] = {};
      for (uint32_t i = 0; i < n; ++i) cnt[e0[i] & 7u]++;
      bool esc = false;
      for (int q = 0; q < 8; ++q) esc = esc || cnt[q] >= 15;
      for (int q = 0; q < 8; ++q) e0[q] |= (esc ? 15u : cnt[q]) << 12;
    }
  }
}

// ------------------------------------------------------------------------------------
// SmoothQuant W8

static void build_w8_image(qlin_layer* L);

static qlin_status build_w8(qlin_layer* L, const float* W, const float* act_absmax) {
  const int N = L->N, K = L->K;
  std::vector<float> aw(K, 0.f);
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) aw[k] = std::max(aw[k], std::fabs(W[(size_t)n * K + k]));
  L->s.resize(K);
  L->s_inv.resize(K);
  const double a = (double)L->alpha;
  for (int k = 0; k < K; ++k) {
    const double num = std::pow(std::max((double)act_absmax[k], 1e-5), a);
    const double den = std::pow(std::max((double)aw[k], 1e-5), 1.0 - a);
    const float sk = (float)(num / den);
    if (!is_finite_f(sk) || sk <= 0.f) return QLIN_ERR_INVALID_ARG;
    L->s[k] = sk;
    L->s_inv[k] = 1.0f / sk;
  }
  L->qw.assign((size_t)N * K, 0);
  L->sw.assign(N, 1.f);
  std::atomic<bool> bad{false};
  parallel_for(N, [&](int64_t b, int64_t e) {
    std::vector<float> ws(K);
    for (int64_t n = b; n < e; ++n) {
      float amax = 0.f;
      for (int k = 0; k < K; ++k) {
        ws[k] = W[(size_t)n * K + k] * L->s[k];
        amax = std::max(amax, std::fabs(ws[k]));
      }
      if (!is_finite_f(amax)) {
        bad = true;
        return;
      }
      const float sc = amax == 0.f ? 1.f : amax / 127.f;
      L->sw[n] = sc;
      for (int k = 0; k < K; ++k) {
        float qv = std::nearbyint(ws[k] / sc);
        qv = std::min(std::max(qv, -127.f), 127.f);
        L->qw[(size_t)n * K + k] = (int8_t)qv;
      }
    }
  });
  if (bad) return QLIN_ERR_INVALID_ARG;
  build_w8_image(L);
  return QLIN_OK;
}

// Device image from the handle's qw, sw and s_inv.
static void build_w8_image(qlin_layer* L) {
  const int N = L->N, K = L->K;
  const int RG = (N + kRowGroup - 1) / kRowGroup, KB = K / kW8Block;
  L->RG = RG;
  L->KU = KB;
  const size_t units_bytes = align256((size_t)RG * KB * kW8UnitBytes);
  const size_t sw_bytes = align256((size_t)RG * kRowGroup * 4);
  const size_t sinv_bytes = align256((size_t)K * 4);
  const int RT = (N + 127) / 128;  // the prefill's 128-row weight tiles
  const size_t w2_bytes = align256((size_t)RT * KB * 4);
  L->sec_units = 0;
  L->sec_sw = units_bytes;
  L->sec_sinv = units_bytes + sw_bytes;
  L->sec_w2 = units_bytes + sw_bytes + sinv_bytes;
  L->image.assign(units_bytes + sw_bytes + sinv_bytes + w2_bytes, 0);
  uint8_t* img = L->image.data();
  parallel_for(RG, [&](int64_t b, int64_t e) {
    for (int64_t rg = b; rg < e; ++rg) {
      for (int kb = 0; kb < KB; ++kb) {
        uint8_t* unit = img + (rg * KB + kb) * kW8UnitBytes;
        for (int rt = 0; rt < 4; ++rt) {
          const int64_t r0 = rg * kRowGroup + rt * 16;
          for (int lane = 0; lane < 32; ++lane) {
            const int gq = lane >> 2, t = lane & 3;
            auto u = [&](int r, int k) -> uint8_t {
              const int64_t n = r0 + r;
              const int v = n < N ? (int)L->qw[(size_t)n * K + k] : 0;
              return (uint8_t)(v + 128);
            };
            for (int j = 0; j < 4; ++j) {  // words 2j, 2j+1: half j / 2, position 2 (j % 2)
              const int k0 = kb * kW8Block + 16 * j;
              uint8_t* w0 = unit + (((size_t)rt * 2 + (j >> 1)) * 32 + lane) * 16 + (j & 1) * 8;
              w0[0] = u(gq, k0 + 2 * t);
              w0[1] = u(gq, k0 + 2 * t + 1);
              w0[2] = u(gq + 8, k0 + 2 * t);
              w0[3] = u(gq + 8, k0 + 2 * t + 1);
              w0[4] = u(gq, k0 + 2 * t + 8);
              w0[5] = u(gq, k0 + 2 * t + 9);
              w0[6] = u(gq + 8, k0 + 2 * t + 8);
              w0[7] = u(gq + 8, k0 + 2 * t + 9);
            }
          }
        }
      }
    }
  });
  float* swd = reinterpret_cast<float*>(img + L->sec_sw);
  for (int n = 0; n < RG * kRowGroup; ++n) swd[n] = n < N ? L->sw[n] : 0.f;
  std::memcpy(img + L->sec_sinv, L->s_inv.data(), (size_t)K * 4);
  // per (128-row tile, 64-wide k-block): the largest sum of squared codes over the tile's rows
  uint32_t* w2 = reinterpret_cast<uint32_t*>(img + L->sec_w2);
  parallel_for(RT, [&](int64_t b, int64_t e) {
    for (int64_t rt = b; rt < e; ++rt)
      for (int kb = 0; kb < KB; ++kb) {
        uint32_t mx = 0;
        for (int64_t n = rt * 128; n < std::min<int64_t>((rt + 1) * 128, N); ++n) {
          const int8_t* q = L->qw.data() + n * K + (int64_t)kb * kW8Block;
          uint32_t s2 = 0;
          for (int k = 0; k < kW8Block; ++k) s2 += (uint32_t)((int)q[k] * (int)q[k]);
          mx = std::max(mx, s2);
        }
        w2[rt * KB + kb] = mx;
      }
  });
}

// ------------------------------------------------------------------------------------
// views for the kernels

static W4View w4view(const qlin_layer* L) {
  return W4View{L->dev + L->sec_units, L->N, L->K, L->RG, L->KU};
}
static SpqrView spqrview(const qlin_layer* L) {
  return SpqrView{L->dev + L->sec_units, reinterpret_cast<const uint32_t*>(L->dev + L->sec_offs),
                  reinterpret_cast<const uint32_t*>(L->dev + L->sec_ents), L->N, L->K, L->RG, L->KU};
}
static W8View w8view(const qlin_layer* L) {
  return W8View{L->dev + L->sec_units, reinterpret_cast<const float*>(L->dev + L->sec_sw),
                reinterpret_cast<const float*>(L->dev + L->sec_sinv), L->N, L->K, L->RG, L->KU,
                reinterpret_cast<const uint32_t*>(L->dev + L->sec_w2)};
}

int qlin_spqr_view_of(qlin_layer* h, SpqrView* out) {
  if (!h || !out || h->format != QLIN_FMT_SPQR) return QLIN_ERR_INVALID_ARG;
  if (!h->dev) return QLIN_ERR_NOT_BOUND;
  *out = spqrview(h);
  return QLIN_OK;
}

// Partial-sum slots the decode launches of a layer may use (one per CTA, or per worker of
// the single-token kernels), for the workspace sizing.
static int decode_grid(const qlin_layer* L) {
  const int64_t units = (int64_t)L->RG * L->KU;
  const int sms = sm_count_cached();
  int64_t g = std::min<int64_t>(units, (int64_t)kMaxCtasPerSm * sms);
  if (L->format == QLIN_FMT_W4G128 || L->format == QLIN_FMT_SPQR)
    g = std::max<int64_t>(g, gemv1_slots(units, sms, L->format == QLIN_FMT_SPQR));
  if (L->format == QLIN_FMT_SPQR) {
    SpqrView v{};
    v.RG = L->RG;
    v.S = L->KU;
    for (int M = 2; M <= 16; ++M) g = std::max<int64_t>(g, spqr_decode_grid(v, M, sms));
  }
  return (int)std::max<int64_t>(1, g);
}

// workspace carve-up
struct WsLayout {
  size_t status, partials, counters, tagged, qx, sx, kbound, total;
};
static WsLayout ws_layout(const qlin_layer* L, int maxM) {
  WsLayout w{};
  const int grid = decode_grid(L);
  w.status = 0;
  w.partials = 256;
  w.counters = w.partials + align256((size_t)grid * 2 * kRowGroup * 16 * 4);
  w.tagged = w.counters + align256((size_t)L->RG * 4);
  w.qx = w.tagged + align256((size_t)grid * 2 * kRowGroup * 4 * 8);
  size_t qx_bytes = 0, sx_bytes = 0;
  if (L->format == QLIN_FMT_W4G128 && !L->perm.empty()) {
    qx_bytes = align256((size_t)std::max(maxM, 1) * L->K * 2);  // act-order: X in permuted channel order
  } else if (L->format == QLIN_FMT_W8A8) {
    // row-major codes for the prefill GEMM, or the decode GEMV's blocked [K/64][M][72] (M <= 16)
    qx_bytes = align256(std::max((size_t)std::max(maxM, 1) * L->K * 2,
                                 (size_t)(L->K / 64) * std::min(std::max(maxM, 1), 16) * 72 * 2));
    sx_bytes = align256((size_t)std::max(maxM, 1) * 4);
  }
  w.sx = w.qx + qx_bytes;
  size_t kb_bytes = 0;
  if (L->format == QLIN_FMT_W8A8) kb_bytes = align256((size_t)((std::max(maxM, 1) + 255) / 256) * (L->K / 64) * 4);
  w.kbound = w.sx + sx_bytes;
  w.total = w.kbound + kb_bytes;
  return w;
}

// ------------------------------------------------------------------------------------
// C ABI

#define QLIN_TRY_ALLOC(expr)                 \
  try {                                      \
    expr;                                    \
  } catch (const std::bad_alloc&) {          \
    return QLIN_ERR_INVALID_ARG;             \
  }

static qlin_status check_w(const float* W, int N, int K) {
  if (!W || N <= 0 || K <= 0) return QLIN_ERR_INVALID_ARG;
  const int64_t total = (int64_t)N * K;
  std::atomic<bool> bad{false};
  parallel_for(total, [&](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i)
      if (!is_finite_f(W[i])) {
        bad = true;
        return;
      }
  });
  return bad ? QLIN_ERR_INVALID_ARG : QLIN_OK;
}

extern "C" {

qlin_status qlin_pack_w4g128(const float* W, int N, int K, qlin_handle* out) {
  if (!out) return QLIN_ERR_INVALID_ARG;
  *out = nullptr;
  if (K % kW4Group) return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_w(W, N, K);
  if (st != QLIN_OK) return st;
  qlin_layer* L = nullptr;
  QLIN_TRY_ALLOC(L = new qlin_layer());
  L->format = QLIN_FMT_W4G128;
  L->N = N;
  L->K = K;
  try {
    st = build_w4(L, W);
  } catch (const std::bad_alloc&) {
    st = QLIN_ERR_INVALID_ARG;
  }
  if (st != QLIN_OK) {
    delete L;
    return st;
  }
  *out = L;
  return QLIN_OK;
}

qlin_status qlin_pack_w4g128_gptq(const float* W, int N, int K, const float* Xcal, int S, double damp,
                                  int act_order, qlin_handle* out) {
  if (!out) return QLIN_ERR_INVALID_ARG;
  *out = nullptr;
  if (K % kW4Group || K > kGptqMaxK || !Xcal || S <= 0 || !(damp > 0.0) || !std::isfinite(damp))
    return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_w(W, N, K);
  if (st != QLIN_OK) return st;
  st = check_w(Xcal, S, K);
  if (st != QLIN_OK) return st;
  qlin_layer* L = nullptr;
  QLIN_TRY_ALLOC(L = new qlin_layer());
  L->format = QLIN_FMT_W4G128;
  L->N = N;
  L->K = K;
  try {
    st = build_w4_gptq(L, W, Xcal, S, damp, act_order != 0);
  } catch (const std::bad_alloc&) {
    st = QLIN_ERR_INVALID_ARG;
  }
  if (st != QLIN_OK) {
    delete L;
    return st;
  }
  *out = L;
  return QLIN_OK;
}

// Checkpoint load: a handle from canonical arrays (the layout qlin_export hands back), checked
// and turned into the same device image a packer writes -- no quantization happens.
static inline bool h_finite(uint16_t h) { return (h & 0x7C00u) != 0x7C00u; }
static inline bool h_small_int(uint16_t h, int maxv) {  // fp16 holding an integer 0..maxv
  const float v = h2f(h);
  return h_finite(h) && v >= 0.f && v <= (float)maxv && std::nearbyint(v) == v && !(h & 0x8000u && v == 0.f);
}
static inline int get_bits3(const uint8_t* stream, size_t row_off, int idx) {
  size_t bit = (size_t)3 * idx;
  int v = 0;
  for (int b = 0; b < 3; ++b, ++bit) v |= ((stream[row_off + bit / 8] >> (bit % 8)) & 1) << b;
  return v;
}

static qlin_status import_w4(qlin_layer* L, const qlin_canonical* c) {
  const int N = L->N, K = L->K, G = K / kW4Group;
  if (!c->codes || !c->scale || !c->zero) return QLIN_ERR_INVALID_ARG;
  for (size_t i = 0; i < (size_t)N * G; ++i) {
    const uint16_t sc = c->scale[i];
    if (!h_finite(sc) || (sc & 0x8000u) || (sc & 0x7FFFu) == 0 || !h_small_int(c->zero[i], 15))
      return QLIN_ERR_INVALID_ARG;
  }
  if (c->perm) {  // act-order: must be a permutation of 0..K-1
    std::vector<uint8_t> seen(K, 0);
    for (int j = 0; j < K; ++j) {
      const int32_t v = c->perm[j];
      if (v < 0 || v >= K || seen[v]) return QLIN_ERR_INVALID_ARG;
      seen[v] = 1;
    }
    L->perm.assign(c->perm, c->perm + K);
  }
  L->scale.assign(c->scale, c->scale + (size_t)N * G);
  L->zero.assign(c->zero, c->zero + (size_t)N * G);
  std::vector<uint8_t> q((size_t)N * K);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n)
      for (int k = 0; k < K; ++k) q[(size_t)n * K + k] = (uint8_t)((c->codes[(size_t)n * (K / 8) + k / 8] >> (4 * (k % 8))) & 15u);
  });
  build_w4_image(L, q);
  return QLIN_OK;
}

static qlin_status import_spqr(qlin_layer* L, const qlin_canonical* c) {
  const int N = L->N, K = L->K, G = K / 16, S = K / kSpqrSuper;
  if (!c->codes3 || !c->qs3 || !c->qz3 || !c->stats || !c->rowptr) return QLIN_ERR_INVALID_ARG;
  if (c->rowptr[0] != 0) return QLIN_ERR_INVALID_ARG;
  for (int n = 0; n < N; ++n) {
    if (c->rowptr[n + 1] < c->rowptr[n] || c->rowptr[n + 1] - c->rowptr[n] > K) return QLIN_ERR_INVALID_ARG;
    for (int32_t p = c->rowptr[n]; p < c->rowptr[n + 1]; ++p) {
      if (!c->col || !c->val) return QLIN_ERR_INVALID_ARG;
      if (c->col[p] < 0 || c->col[p] >= K || (p > c->rowptr[n] && c->col[p] <= c->col[p - 1])) return QLIN_ERR_INVALID_ARG;
      if (!h_finite(c->val[p])) return QLIN_ERR_INVALID_ARG;
    }
  }
  for (size_t i = 0; i < (size_t)N * S; ++i) {
    const uint16_t* st = c->stats + 4 * i;
    if (!h_finite(st[0]) || !h_finite(st[2]) || !h_small_int(st[1], 7) || !h_small_int(st[3], 7))
      return QLIN_ERR_INVALID_ARG;
  }
  const int64_t nnz = c->rowptr[N];
  L->nnz = nnz;
  L->frac = (float)((double)nnz / ((double)N * K));
  L->stats.assign(c->stats, c->stats + (size_t)N * S * 4);
  L->rowptr.assign(c->rowptr, c->rowptr + N + 1);
  L->col.assign(c->col ? c->col : nullptr, c->col ? c->col + nnz : nullptr);
  L->val.assign(c->val ? c->val : nullptr, c->val ? c->val + nnz : nullptr);
  const size_t cb = (size_t)3 * K / 8, sb = (size_t)3 * G / 8;
  L->codes3.assign(c->codes3, c->codes3 + (size_t)N * cb);
  L->qs3.assign(c->qs3, c->qs3 + (size_t)N * sb);
  L->qz3.assign(c->qz3, c->qz3 + (size_t)N * sb);
  std::vector<uint8_t> q((size_t)N * K), qs((size_t)N * G), qz((size_t)N * G);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n) {
      for (int k = 0; k < K; ++k) q[(size_t)n * K + k] = (uint8_t)get_bits3(c->codes3, n * cb, k);
      for (int g = 0; g < G; ++g) {
        qs[(size_t)n * G + g] = (uint8_t)get_bits3(c->qs3, n * sb, g);
        qz[(size_t)n * G + g] = (uint8_t)get_bits3(c->qz3, n * sb, g);
      }
    }
  });
  build_spqr_image(L, q, qs, qz);
  return QLIN_OK;
}

static qlin_status import_w8(qlin_layer* L, const qlin_canonical* c) {
  const int N = L->N, K = L->K;
  if (!c->qw || !c->sw || !c->s || !c->s_inv) return QLIN_ERR_INVALID_ARG;
  for (size_t i = 0; i < (size_t)N * K; ++i)
    if (c->qw[i] < -127) return QLIN_ERR_INVALID_ARG;
  for (int n = 0; n < N; ++n)
    if (!is_finite_f(c->sw[n]) || !(c->sw[n] > 0.f)) return QLIN_ERR_INVALID_ARG;
  for (int k = 0; k < K; ++k)
    if (!is_finite_f(c->s[k]) || !(c->s[k] > 0.f) || !is_finite_f(c->s_inv[k]) || !(c->s_inv[k] > 0.f))
      return QLIN_ERR_INVALID_ARG;
  L->qw.assign(c->qw, c->qw + (size_t)N * K);
  L->sw.assign(c->sw, c->sw + N);
  L->s.assign(c->s, c->s + K);
  L->s_inv.assign(c->s_inv, c->s_inv + K);
  build_w8_image(L);
  return QLIN_OK;
}

qlin_status qlin_import(int format, int N, int K, const qlin_canonical* in, qlin_handle* out) {
  if (!out) return QLIN_ERR_INVALID_ARG;
  *out = nullptr;
  if (!in || N <= 0 || K <= 0) return QLIN_ERR_INVALID_ARG;
  if (format == QLIN_FMT_W4G128 && K % kW4Group) return QLIN_ERR_INVALID_ARG;
  if (format == QLIN_FMT_SPQR && (K % kSpqrSuper || K > 32768)) return QLIN_ERR_INVALID_ARG;
  if (format == QLIN_FMT_W8A8 && K % kW8Block) return QLIN_ERR_INVALID_ARG;
  if (format != QLIN_FMT_W4G128 && format != QLIN_FMT_SPQR && format != QLIN_FMT_W8A8) return QLIN_ERR_INVALID_ARG;
  qlin_layer* L = nullptr;
  QLIN_TRY_ALLOC(L = new qlin_layer());
  L->format = format;
  L->N = N;
  L->K = K;
  qlin_status st = QLIN_ERR_INVALID_ARG;
  try {
    st = format == QLIN_FMT_W4G128 ? import_w4(L, in) : format == QLIN_FMT_SPQR ? import_spqr(L, in) : import_w8(L, in);
  } catch (const std::bad_alloc&) {
    st = QLIN_ERR_INVALID_ARG;
  }
  if (st != QLIN_OK) {
    delete L;
    return st;
  }
  *out = L;
  return QLIN_OK;
}

qlin_status qlin_pack_spqr(const float* W, int N, int K, float outlier_frac, qlin_handle* out) {
  if (!out) return QLIN_ERR_INVALID_ARG;
  *out = nullptr;
  if (K % kSpqrSuper || K > 32768) return QLIN_ERR_INVALID_ARG;
  if (!(outlier_frac >= 0.f && outlier_frac < 1.f)) return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_w(W, N, K);
  if (st != QLIN_OK) return st;
  qlin_layer* L = nullptr;
  QLIN_TRY_ALLOC(L = new qlin_layer());
  L->format = QLIN_FMT_SPQR;
  L->N = N;
  L->K = K;
  L->frac = outlier_frac;
  try {
    st = build_spqr(L, W);
  } catch (const std::bad_alloc&) {
    st = QLIN_ERR_INVALID_ARG;
  }
  if (st != QLIN_OK) {
    delete L;
    return st;
  }
  *out = L;
  return QLIN_OK;
}

qlin_status qlin_pack_w8(const float* W, int N, int K, const float* act_absmax, float alpha,
                         qlin_handle* out) {
  if (!out) return QLIN_ERR_INVALID_ARG;
  *out = nullptr;
  if (!act_absmax || K % kW8Block) return QLIN_ERR_INVALID_ARG;
  if (!(alpha >= 0.f && alpha <= 1.f)) return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_w(W, N, K);
  if (st != QLIN_OK) return st;
  for (int k = 0; k < K; ++k)
    if (!is_finite_f(act_absmax[k]) || act_absmax[k] < 0.f) return QLIN_ERR_INVALID_ARG;
  qlin_layer* L = nullptr;
  QLIN_TRY_ALLOC(L = new qlin_layer());
  L->format = QLIN_FMT_W8A8;
  L->N = N;
  L->K = K;
  L->alpha = alpha;
  try {
    st = build_w8(L, W, act_absmax);
  } catch (const std::bad_alloc&) {
    st = QLIN_ERR_INVALID_ARG;
  }
  if (st != QLIN_OK) {
    delete L;
    return st;
  }
  *out = L;
  return QLIN_OK;
}

qlin_status qlin_device_bytes(qlin_handle h, size_t* weight_bytes) {
  if (!h || !weight_bytes) return QLIN_ERR_INVALID_ARG;
  *weight_bytes = h->image.size();
  return QLIN_OK;
}

qlin_status qlin_workspace_bytes(qlin_handle h, int max_M, size_t* bytes) {
  if (!h || !bytes || max_M < 0) return QLIN_ERR_INVALID_ARG;
  *bytes = ws_layout(h, max_M).total;
  return QLIN_OK;
}

qlin_status qlin_bind(qlin_handle h, void* dev_weights, size_t bytes, qlin_stream stream) {
  if (!h || !dev_weights) return QLIN_ERR_INVALID_ARG;
  if (bytes < h->image.size() || ((uintptr_t)dev_weights & 255u)) return QLIN_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(dev_weights, h->image.data(), h->image.size(),
                                  cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return QLIN_ERR_CUDA;
  h->dev = (uint8_t*)dev_weights;
  h->dev_bytes = bytes;
  // the allocation-free SpQR forward's scratch array goes onto the device now, while device
  // memory is free (best effort: qlin_forward_spqr_static reports a failure itself)
  if (h->format == QLIN_FMT_SPQR) qlin_static_scratch_prepare();
  return QLIN_OK;
}

qlin_status qlin_attach(qlin_handle h, void* dev_weights, size_t bytes) {
  if (!h || !dev_weights) return QLIN_ERR_INVALID_ARG;
  if (bytes < h->image.size() || ((uintptr_t)dev_weights & 255u)) return QLIN_ERR_INVALID_ARG;
  h->dev = (uint8_t*)dev_weights;
  h->dev_bytes = bytes;
  if (h->format == QLIN_FMT_SPQR) qlin_static_scratch_prepare();  // as in qlin_bind
  return QLIN_OK;
}

qlin_status qlin_set_workspace(qlin_handle h, void* dev_ws, size_t bytes, int max_M, qlin_stream stream) {
  if (!h || !dev_ws || max_M < 0 || ((uintptr_t)dev_ws & 255u)) return QLIN_ERR_INVALID_ARG;
  WsLayout w = ws_layout(h, max_M);
  if (bytes < w.total) return QLIN_ERR_WORKSPACE;
  // status word, partial slots and counters start at zero; counters return to zero after
  // every forward (the last contributor of a row group resets its counter)
  if (cudaMemsetAsync(dev_ws, 0, w.qx, (cudaStream_t)stream) != cudaSuccess) return QLIN_ERR_CUDA;
  for (auto& g : h->host_graphs) cudaGraphExecDestroy(g.exec);  // they hold the old workspace
  h->host_graphs.clear();
  h->ws = (uint8_t*)dev_ws;
  h->ws_bytes = bytes;
  h->ws_maxM = max_M;
  h->grid = decode_grid(h);
  h->wsv.status = reinterpret_cast<int32_t*>(h->ws + w.status);
  h->wsv.partials = reinterpret_cast<float*>(h->ws + w.partials);
  h->wsv.counters = reinterpret_cast<uint32_t*>(h->ws + w.counters);
  h->wsv.tagged = reinterpret_cast<uint64_t*>(h->ws + w.tagged);
  h->wsv.tag = 1u;
  h->wsv.qx = h->ws + w.qx;
  h->wsv.sx = reinterpret_cast<float*>(h->ws + w.sx);
  h->wsv.kbound = reinterpret_cast<int32_t*>(h->ws + w.kbound);
  h->wsv.grid = h->grid;
  h->wsv.sms = sm_count_cached();
  return QLIN_OK;
}

static qlin_status check_forward(qlin_handle h, const void* X, const void* Y, int M) {
  if (!h || M < 0) return QLIN_ERR_INVALID_ARG;
  if (M == 0) return QLIN_OK;
  if (!X || !Y || ((uintptr_t)X & 15u) || ((uintptr_t)Y & 15u)) return QLIN_ERR_INVALID_ARG;
  if (!h->dev) return QLIN_ERR_NOT_BOUND;
  if (!h->ws || ((h->format == QLIN_FMT_W8A8 || !h->perm.empty()) && M > h->ws_maxM)) return QLIN_ERR_WORKSPACE;
  return QLIN_OK;
}

static qlin_status run_decode(qlin_handle h, const uint16_t* X, uint16_t* Y, int32_t* acc, int M,
                              cudaStream_t s) {
  int e = 0;
  switch (h->format) {
    case QLIN_FMT_W4G128: {
      W4View v = w4view(h);
      if (!h->perm.empty()) {  // act-order: x's channels are read in the permuted order
        const int32_t* perm = reinterpret_cast<const int32_t*>(h->dev + h->sec_perm);
        if (M == 1 && h->K <= kG1GatherMaxK) {
          v.perm = perm;  // the single-token kernel gathers x while staging it
        } else {          // a gather launch first
          uint16_t* xp = reinterpret_cast<uint16_t*>(h->wsv.qx);
          e = launch_w4_gather(X, perm, xp, M, h->K, s);
          X = xp;
        }
      }
      if (!e) e = launch_w4_decode(v, X, Y, M, h->wsv, h->grid, s);
      break;
    }
    case QLIN_FMT_SPQR:
      e = launch_spqr_decode(spqrview(h), X, Y, M, h->wsv, h->grid, s);
      break;
    case QLIN_FMT_W8A8: {
      uint16_t* q16 = reinterpret_cast<uint16_t*>(h->wsv.qx);
      e = launch_w8_act_quant_f16(w8view(h), X, q16, h->wsv.sx, nullptr, M, true, s);
      if (!e) e = launch_w8_decode(w8view(h), q16, h->wsv.sx, Y, acc, M, h->wsv, h->grid, s);
      break;
    }
    default:
      return QLIN_ERR_INVALID_ARG;
  }
  return e ? QLIN_ERR_CUDA : QLIN_OK;
}

// Prefill (M > 16): tensor-core kernels, one launch (two for W8A8: act-quant + GEMM).
static qlin_status run_prefill(qlin_handle h, const uint16_t* X, uint16_t* Y, int32_t* acc, int M, cudaStream_t s) {
  int e = 0;
  switch (h->format) {
    case QLIN_FMT_W4G128:
      if (!h->perm.empty()) {
        uint16_t* xp = reinterpret_cast<uint16_t*>(h->wsv.qx);
        e = launch_w4_gather(X, reinterpret_cast<const int32_t*>(h->dev + h->sec_perm), xp, M, h->K, s);
        X = xp;
      }
      if (!e) e = launch_w4_prefill(w4view(h), X, Y, M, h->wsv.status, s);
      break;
    case QLIN_FMT_SPQR:
      e = launch_spqr_prefill(spqrview(h), X, Y, M, h->wsv.status, s);
      break;
    case QLIN_FMT_W8A8: {
      uint16_t* q16 = reinterpret_cast<uint16_t*>(h->wsv.qx);
      // per-tile bounds of sum |qx| per k-block, gathered by the act-quant kernel with atomicMax
      const size_t kb_bytes = (size_t)((M + 255) / 256) * (h->K / 64) * 4;
      e = (int)cudaMemsetAsync(h->wsv.kbound, 0, kb_bytes, s);
      if (!e) e = launch_w8_act_quant_f16(w8view(h), X, q16, h->wsv.sx, h->wsv.kbound, M, false, s);
      if (!e) e = launch_w8_prefill(w8view(h), q16, h->wsv.sx, h->wsv.kbound, Y, acc, M, h->wsv.status, s);
      break;
    }
    default:
      return QLIN_ERR_INVALID_ARG;
  }
  return e ? QLIN_ERR_CUDA : QLIN_OK;
}

qlin_status qlin_forward(qlin_handle h, const void* X, void* Y, int M, qlin_stream stream) {
  qlin_status st = check_forward(h, X, Y, M);
  if (st != QLIN_OK || M == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (M > 16) return run_prefill(h, (const uint16_t*)X, (uint16_t*)Y, nullptr, M, s);
  return run_decode(h, (const uint16_t*)X, (uint16_t*)Y, nullptr, M, s);
}

// The step's three stream operations, enqueued on s.
static qlin_status host_step(qlin_handle h, const void* X_host, void* Y_host, void* X_dev, void* Y_dev, int M,
                             cudaStream_t s) {
  if (cudaMemcpyAsync(X_dev, X_host, (size_t)M * h->K * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return QLIN_ERR_CUDA;
  qlin_status st = qlin_forward(h, X_dev, Y_dev, M, (qlin_stream)s);
  if (st != QLIN_OK) return st;
  if (cudaMemcpyAsync(Y_host, Y_dev, (size_t)M * h->N * 2, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QLIN_ERR_CUDA;
  return QLIN_OK;
}

static constexpr size_t kMaxHostGraphs = 64;

// The step as one CUDA graph launch: captured the first time a set of pointers, M and stream is
// seen (the copies, the kernels and their programmatic dependencies baked in), replayed after.
// Returns QLIN_ERR_UNSUPPORTED (nothing enqueued) where capture is not possible.
static qlin_status host_step_graph(qlin_handle h, const void* X_host, void* Y_host, void* X_dev, void* Y_dev, int M,
                                   cudaStream_t s) {
  if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread) return QLIN_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return QLIN_ERR_UNSUPPORTED;
  ++h->host_graph_clock;
  for (auto& g : h->host_graphs) {
    if (g.xh == X_host && g.yh == Y_host && g.xd == X_dev && g.yd == Y_dev && g.dev == h->dev && g.M == M &&
        g.stream == s) {
      g.used = h->host_graph_clock;
      return cudaGraphLaunch(g.exec, s) == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA;
    }
  }
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return QLIN_ERR_UNSUPPORTED;
  }
  const qlin_status st = host_step(h, X_host, Y_host, X_dev, Y_dev, M, s);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  if (st != QLIN_OK || ec != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return st != QLIN_OK ? st : QLIN_ERR_UNSUPPORTED;
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess || !exec) {
    cudaGetLastError();
    return QLIN_ERR_UNSUPPORTED;
  }
  if (h->host_graphs.size() >= kMaxHostGraphs) {  // drop the least recently used
    size_t lru = 0;
    for (size_t i = 1; i < h->host_graphs.size(); ++i)
      if (h->host_graphs[i].used < h->host_graphs[lru].used) lru = i;
    cudaGraphExecDestroy(h->host_graphs[lru].exec);
    h->host_graphs.erase(h->host_graphs.begin() + (ptrdiff_t)lru);
  }
  h->host_graphs.push_back(HostGraph{X_host, Y_host, X_dev, Y_dev, h->dev, M, s, exec, h->host_graph_clock});
  return cudaGraphLaunch(exec, s) == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA;
}

qlin_status qlin_forward_host(qlin_handle h, const void* X_host, void* Y_host, void* X_dev,
                              void* Y_dev, int M, qlin_stream stream) {
  if (!X_host || !Y_host) return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_forward(h, X_dev, Y_dev, M);
  if (st != QLIN_OK || M == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  st = host_step_graph(h, X_host, Y_host, X_dev, Y_dev, M, s);
  if (st == QLIN_ERR_UNSUPPORTED) st = host_step(h, X_host, Y_host, X_dev, Y_dev, M, s);
  if (st != QLIN_OK) return st;
  return cudaStreamSynchronize(s) == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA;
}

qlin_status qlin_act_quant(qlin_handle h, const void* X, int8_t* qx, float* sx, int M, qlin_stream stream) {
  if (!h || h->format != QLIN_FMT_W8A8 || M < 0) return QLIN_ERR_INVALID_ARG;
  if (M == 0) return QLIN_OK;
  if (!X || !qx || !sx || ((uintptr_t)X & 15u)) return QLIN_ERR_INVALID_ARG;
  if (!h->dev) return QLIN_ERR_NOT_BOUND;
  int e = launch_w8_act_quant(w8view(h), (const uint16_t*)X, qx, sx, M, (cudaStream_t)stream);
  return e ? QLIN_ERR_CUDA : QLIN_OK;
}

qlin_status qlin_forward_acc(qlin_handle h, const void* X, int32_t* acc, int M, qlin_stream stream) {
  if (!h || h->format != QLIN_FMT_W8A8) return QLIN_ERR_INVALID_ARG;
  qlin_status st = check_forward(h, X, acc, M);
  if (st != QLIN_OK || M == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (M > 16) return run_prefill(h, (const uint16_t*)X, nullptr, acc, M, s);
  return run_decode(h, (const uint16_t*)X, nullptr, acc, M, s);
}

qlin_status qlin_dequant_device(qlin_handle h, void* out, qlin_stream stream) {
  if (!h || !out) return QLIN_ERR_INVALID_ARG;
  if (!h->dev) return QLIN_ERR_NOT_BOUND;
  int e = 0;
  cudaStream_t s = (cudaStream_t)stream;
  switch (h->format) {
    case QLIN_FMT_W4G128: e = launch_w4_dequant(w4view(h), (float*)out, s); break;
    case QLIN_FMT_SPQR: e = launch_spqr_dequant(spqrview(h), (float*)out, s); break;
    case QLIN_FMT_W8A8: e = launch_w8_export(w8view(h), (int8_t*)out, s); break;
    default: return QLIN_ERR_INVALID_ARG;
  }
  return e ? QLIN_ERR_CUDA : QLIN_OK;
}

qlin_status qlin_poll_status(qlin_handle h, qlin_stream stream) {
  if (!h) return QLIN_ERR_INVALID_ARG;
  if (!h->ws) return QLIN_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QLIN_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, h->wsv.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return QLIN_ERR_CUDA;
  if (v != 0) {
    const int32_t zero = 0;
    if (cudaMemcpy(h->wsv.status, &zero, 4, cudaMemcpyHostToDevice) != cudaSuccess) return QLIN_ERR_CUDA;
    return v == kStatusTimeout ? QLIN_ERR_TIMEOUT : QLIN_ERR_CUDA;
  }
  return QLIN_OK;
}

qlin_status qlin_export(qlin_handle h, qlin_canonical* o) {
  if (!h || !o) return QLIN_ERR_INVALID_ARG;
  std::memset(o, 0, sizeof(*o));
  auto p = [](const auto& v) { return v.empty() ? nullptr : v.data(); };
  o->codes = p(h->codes);
  o->scale = p(h->scale);
  o->zero = p(h->zero);
  o->codes3 = p(h->codes3);
  o->qs3 = p(h->qs3);
  o->qz3 = p(h->qz3);
  o->stats = p(h->stats);
  o->rowptr = p(h->rowptr);
  o->col = p(h->col);
  o->val = p(h->val);
  o->qw = p(h->qw);
  o->sw = p(h->sw);
  o->s = p(h->s);
  o->s_inv = p(h->s_inv);
  o->perm = p(h->perm);
  return QLIN_OK;
}

qlin_status qlin_info(qlin_handle h, qlin_layer_info* o) {
  if (!h || !o) return QLIN_ERR_INVALID_ARG;
  std::memset(o, 0, sizeof(*o));
  o->format = h->format;
  o->N = h->N;
  o->K = h->K;
  o->nnz = h->nnz;
  const int64_t N = h->N, K = h->K;
  int64_t pb = 0;
  switch (h->format) {
    case QLIN_FMT_W4G128: pb = N * K / 2 + N * (K / kW4Group) * 4 + 4 * (int64_t)h->perm.size(); break;
    case QLIN_FMT_SPQR:
      pb = N * (3 * K / 8) + 2 * N * (3 * (K / 16) / 8) + N * (K / kSpqrSuper) * 8 + 4 * (N + 1) + 4 * h->nnz;
      break;
    case QLIN_FMT_W8A8: pb = N * K + 4 * N + 4 * K; break;
  }
  o->packed_bytes = pb;
  o->bits_per_param = 8.0 * (double)pb / (double)(N * K);
  o->device_bytes = (int64_t)h->image.size();
  o->alpha = h->alpha;
  o->outlier_frac = h->frac;
  return QLIN_OK;
}

void qlin_destroy(qlin_handle h) { delete h; }

const char* qlin_status_string(qlin_status s) {
  switch (s) {
    case QLIN_OK: return "ok";
    case QLIN_ERR_INVALID_ARG: return "invalid argument";
    case QLIN_ERR_UNSUPPORTED: return "unsupported";
    case QLIN_ERR_CUDA: return "CUDA error";
    case QLIN_ERR_WORKSPACE: return "workspace missing or too small";
    case QLIN_ERR_TIMEOUT: return "device-side wait timed out";
    case QLIN_ERR_NOT_BOUND: return "weights not bound to device memory";
  }
  return "unknown status";
}

int qlin_sm_count(void) { return sm_count_cached(); }

qlin_status qlin_debug_wait_timeout(int32_t* status, int limit_us, qlin_stream stream) {
  if (!status || limit_us <= 0 || limit_us > 10000000) return QLIN_ERR_INVALID_ARG;
  return launch_debug_wait_timeout(status, limit_us, stream) ? QLIN_ERR_CUDA : QLIN_OK;
}

}  // extern "C"

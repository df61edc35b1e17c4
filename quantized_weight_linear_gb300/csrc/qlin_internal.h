// Internal declarations shared by the host library and the CUDA kernels.
//
// Device weight images.  Every format is cut into "units": a row group of 64 output
// rows (four row tiles of 16, one per consumer warp) times a K chunk.  Units are stored
// contiguously in row-group-major order, so that any contiguous range of units is one
// contiguous byte range (a decode CTA streams such a range with bulk copies).  Rows past
// N are zero padding and are never stored to Y.
//
// W4G128 unit = (row group, one 128-wide K group), 4352 bytes:
//   codes  [4 row tiles][2 k-blocks of 64][32 lanes][4 words]      4096 B
//   stats  [4 row tiles][16 rows] (scale fp16, zero fp16)            256 B
//   For row tile rt, k-block kb, lane l = 4g + t, word j (k16 tile k0 = 64 kb + 16 j):
//   nibble 0 = q[g][k0+2t]   nibble 4 = q[g][k0+2t+1]
//   nibble 1 = q[g+8][k0+2t] nibble 5 = q[g+8][k0+2t+1]
//   nibble 2 = q[g][k0+2t+8] nibble 6 = q[g][k0+2t+9]
//   nibble 3 = q[g+8][k0+2t+8] nibble 7 = q[g+8][k0+2t+9]
//   (rows relative to the tile) -- the A-fragment order of an m16n8k16 MMA, so that
//   ((w >> 4r) & 0x000F000F) | 0x43004300 is A register r as bf16 pairs (128 + q).
//
// SPQR unit = (row group, one 256-wide supergroup = 2 blocks of 128), 7424 bytes:
//   codes  [4 row tiles][2 blocks][32 lanes][6 words]               6144 B
//   qsqz   [4 row tiles][2 blocks][32 lanes] 24-bit fields, packed    768 B
//   sgst   [4 row tiles][16 rows][4 fp16] (ss, zs, sz, zz)            512 B
//   In a block (16 rows x 8 groups of 16), lane (g, t) owns the A-fragment pairs of
//   (row g, group t), (row g+8, group t), (row g, group t+4), (row g+8, group t+4); MMA j
//   (0..7) consumes elements 2j, 2j+1 of each.  A 32-bit code word holds 10 codes as two
//   halves of five 3-bit fields (bits 0,3,6,9,12 of each half, bit 15 spare):
//     pair index i = 4j + r, j <= 4: word i/3, field (0, 2, 4)[i % 3] (bf16 base 128);
//                              i in {18, 19}: spare bits of words 3(i-18) .. 3(i-18)+2
//                              (bit 15 -> code bit 0,1,2 in word order; bit 31 likewise)
//     pair index i = 4(j-5) + r, j >= 5: word i/2, field (1, 3)[i % 2] (bf16 base 16).
//   The low half holds element 2j, the high half element 2j+1.
//   qsqz: lane (g, t) owns a 24-bit field at bit 24*lane of the block's 96 bytes:
//     bits [6i, 6i+3) qs, [6i+3, 6i+6) qz of pair i = (row g, group 2t), (row g, group 2t+1),
//     (row g+8, group 2t), (row g+8, group 2t+1)  -- the accumulator (C) side of the MMA.
//   Outliers: a separate entry array of uint32 (fp16 value << 16 | k in unit << 4 | row
//   in tile), bucketed by (unit, row tile); offs[(unit * 4 + rt)] is the first entry of a
//   bucket and offs[units * 4] the total.  Within a bucket entries are sorted by quad
//   (row & 7), then row, then k: the rows g and g + 8 of MMA lane quad g form one run, each
//   row a run inside it.  Bits 12..15 of entries 0..7 of a bucket with at least 8 entries
//   hold the entry counts of quads 0..7, or 15 in all eight when a quad has 15 or more
//   (bits 12..15 of every other entry are zero).
//
// W8A8 unit = (row group, one 64-wide K block), 4096 bytes of codes:
//   codes [4 row tiles][2 halves][32 lanes][4 words] bytes u = q + 128 in A-fragment order
//   (a lane's 8 words split in two halves of 16 bytes, so that a warp's 16-byte loads of a
//   half are contiguous); lane word w (0..7) sits in half w / 4 at position w % 4; for
//   k16 tile j: word 2j = (row g k 2t, row g k 2t+1, row g+8 k 2t, row g+8 k 2t+1),
//   word 2j+1 = the same at k 2t+8, 2t+9; plus per-row fp32 sw and per-channel fp32
//   s_inv in their own sections.
#pragma once
#include <cstddef>
#include <cstdint>

namespace qlin {

constexpr int kRowGroup = 64;     // rows per unit (4 row tiles x 16)
constexpr int kW4Group = 128;
constexpr int kW4UnitBytes = 4352;
constexpr int kW4CodeBytes = 4096;
constexpr int kSpqrSuper = 256;
constexpr int kSpqrUnitBytes = 7424;
constexpr int kSpqrCodeBytes = 6144;
constexpr int kSpqrQsqzBytes = 768;
constexpr int kW8Block = 64;
constexpr int kW8UnitBytes = 4096;

// device status word values (first int32 of the workspace)
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 5;

struct W4View {
  const uint8_t* units;  // [RG][G] units
  int N, K, RG, G;
  // act-order column permutation, when the single-token kernel gathers x itself (M == 1,
  // K <= kG1GatherMaxK); otherwise null and x arrives already permuted
  const int32_t* perm = nullptr;
};
#ifndef QLIN_G1_GATHER_MAX_K
#define QLIN_G1_GATHER_MAX_K 8192
#endif
constexpr int kG1GatherMaxK = QLIN_G1_GATHER_MAX_K;

struct SpqrView {
  const uint8_t* units;      // [RG][S] units
  const uint32_t* offs;      // [RG*S*4 + 1]
  const uint32_t* ents;      // [nnz]
  int N, K, RG, S;
};

struct W8View {
  const uint8_t* units;  // [RG][K/64] units
  const float* sw;       // [Npad]
  const float* s_inv;    // [K]
  int N, K, RG, KB;
  // [ceil(N / 128)][K / 64]: max over a 128-row tile of sum qw^2 over a 64-wide k-block (the
  // prefill's exact-chunk bounds)
  const uint32_t* w2;
};

// Workspace carve-up (all offsets 256-byte aligned).
struct Workspace {
  int32_t* status;     // device status word
  float* partials;     // [grid][2][64 * 16] split-row partial sums
  uint32_t* counters;  // [RG] arrival counters of split row groups
  uint64_t* tagged;    // [grid][2][64 * 4] partial sums of up to 4 tokens as 8-byte words (value, tag)
  uint32_t tag;        // nonzero tag of this workspace's valid words in `tagged`
  void* qx;            // W8A8: fp16 activation codes [maxM][K]
  float* sx;           // W8A8: [maxM]
  int32_t* kbound;     // W8A8 prefill: [ceil(maxM / 256)][K / 64] max over a 256-token tile of
                       // sum qx^2 over a 64-wide k-block (sizes the exact fp32 chunks)
  int grid;            // largest decode grid the partial slots were sized for
  int sms;             // SM count of the device
};

constexpr int kMaxCtasPerSm = 4;  // decode kernels run up to 4 CTAs per SM

// ---- kernel launchers (kern_*.cu); all asynchronous, return cudaError_t as int ----
int launch_w4_decode(const W4View& v, const uint16_t* X, uint16_t* Y, int M, const Workspace& ws,
                     int grid, void* stream);
// act-order W4: Xp[m][j] = X[m][perm[j]] (K % 8 == 0, 16-byte aligned rows)
int launch_w4_gather(const uint16_t* X, const int32_t* perm, uint16_t* Xp, int M, int K, void* stream);
int launch_spqr_decode(const SpqrView& v, const uint16_t* X, uint16_t* Y, int M,
                       const Workspace& ws, int grid, void* stream);
int launch_w8_act_quant(const W8View& v, const uint16_t* X, int8_t* qx, float* sx, int M,
                        void* stream);
// blocked: codes laid out [K/64][M][72] for the decode GEMV (M <= 16) instead of [M][K]
int launch_w8_act_quant_f16(const W8View& v, const uint16_t* X, uint16_t* q16, float* sx, int32_t* kbound, int M,
                            bool blocked, void* stream);
int launch_w8_decode(const W8View& v, const uint16_t* q16, const float* sx, uint16_t* Y,
                     int32_t* acc_out, int M, const Workspace& ws, int grid, void* stream);
int launch_w4_prefill(const W4View& v, const uint16_t* X, uint16_t* Y, int M, int32_t* status, void* stream);
int launch_spqr_prefill(const SpqrView& v, const uint16_t* X, uint16_t* Y, int M, int32_t* status,
                        void* stream);
int launch_w8_prefill(const W8View& v, const uint16_t* q16, const float* sx, const int32_t* kbound, uint16_t* Y,
                      int32_t* acc, int M, int32_t* status, void* stream);
int spqr_decode_grid(const SpqrView& v, int M, int sms);
// Single-token (M == 1) decode of W4 and SpQR (kern_gemv1.cu); the multi-token launchers
// above hand M == 1 to these.  gemv1_slots: partial-sum slots (workers) such a launch uses.
int launch_spqr_gemv1(const SpqrView& v, const uint16_t* X, uint16_t* Y, const Workspace& ws, void* stream);
int launch_w4_gemv1(const W4View& v, const uint16_t* X, uint16_t* Y, const Workspace& ws, void* stream);
int gemv1_slots(int64_t units, int sms, bool spqr);
// Loads the allocation-free SpQR forward's fixed scratch array on the current device
// (kern_static_ws.cu); returns a qlin_status.
int qlin_static_scratch_prepare();

}  // namespace qlin

// The SpQR device view of a bound handle: QLIN_OK, QLIN_ERR_INVALID_ARG (another format)
// or QLIN_ERR_NOT_BOUND.  Defined with the handle in qlin_host.cpp.
struct qlin_layer;
int qlin_spqr_view_of(struct qlin_layer* h, qlin::SpqrView* out);

namespace qlin {
int launch_w4_dequant(const W4View& v, float* out, void* stream);
int launch_spqr_dequant(const SpqrView& v, float* out, void* stream);
int launch_w8_export(const W8View& v, int8_t* out, void* stream);
int launch_debug_wait_timeout(int32_t* status, int limit_us, void* stream);

}  // namespace qlin

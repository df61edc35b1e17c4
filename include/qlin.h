/*
 * qlin -- quantized linear-layer forward Y = X . W_hat^T on one GB300 (sm_103a).
 *
 * C ABI: plain pointers and sizes; no C++ types, no exceptions across the boundary.
 *
 * Formats (the operation each one defines):
 *
 *  W4G128   GPTQ page ("Makale Bülteni — GPTQ"), sections "İddia ve Gerçeklik: GPTQ"
 *           (4-bit weights quantized in groups, 128 given as the block size; weight-only,
 *           activations stay 16-bit) and the intro (round-to-nearest as the baseline
 *           quantizer).  Codes uint4, 8 per uint32, fp16 scale and zero per (row, 128-wide
 *           K group):  w_hat = (q - z) * s.
 *  SPQR     SpQR page ("Makale Bülteni — SpQR"), section "İddia ve Gerçeklik: SpQR":
 *           W_hat = D + S, D a 3-bit dense matrix in groups of 16 whose per-group scales
 *           and zeros are themselves 3-bit codes under fp16 statistics per 16 groups
 *           (bi-level), S about 1% of the entries kept as fp16 in a sparse matrix, applied
 *           in the same pass as the dense unpack.
 *  W8A8     SmoothQuant page ("Makale Bülteni — SmoothQuant"), section "İddia ve
 *           Gerçeklik: SmoothQuant": Y = (X diag(s)^-1)(diag(s) W), s folded into W
 *           offline, X quantized per token and W per output channel to int8, integer
 *           accumulation, scale epilogue y = bf16((acc * sx_m) * sw_n).
 *
 * Shapes and layouts: X is bf16 [M][K] row-major, Y is bf16 [M][N] row-major, W (the
 * fp32 matrix handed to a packer) is [N][K] row-major (out x in).  Groups run along K.
 *
 * Memory ownership: the library never allocates device memory.  The caller (in the
 * Python binding: PyTorch) allocates the weight image, the workspace, X and Y and keeps
 * them alive while any call that uses them is in flight.  Handles own only host memory.
 *
 * Errors: every call returns a qlin_status.  Asynchronous calls report argument and
 * launch errors only; a device-side wait that ran out of its limit is reported by
 * qlin_poll_status.  A handle is not safe for concurrent qlin_bind / qlin_set_workspace;
 * forwards on one handle must not overlap on the GPU (they share the workspace).
 */
#ifndef QLIN_H_
#define QLIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLIN_OK = 0,
  QLIN_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer, non-finite input */
  QLIN_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  QLIN_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  QLIN_ERR_WORKSPACE = 4,   /* workspace missing or smaller than qlin_workspace_bytes */
  QLIN_ERR_TIMEOUT = 5,     /* a device-side wait gave up after its time limit (2 s) */
  QLIN_ERR_NOT_BOUND = 6    /* forward on a handle whose weights were never bound */
} qlin_status;

typedef enum { QLIN_FMT_W4G128 = 1, QLIN_FMT_SPQR = 2, QLIN_FMT_W8A8 = 3 } qlin_format;

/* Opaque layer handle (host object). */
typedef struct qlin_layer* qlin_handle;

/* CUDA stream as an opaque pointer (a cudaStream_t; NULL = legacy default stream). */
typedef void* qlin_stream;

typedef struct {
  int32_t format;          /* qlin_format */
  int32_t N, K;
  int64_t nnz;             /* SpQR outliers (0 otherwise) */
  int64_t packed_bytes;    /* canonical packed size: codes + statistics (+ CSR) */
  double bits_per_param;   /* 8 * packed_bytes / (N * K) */
  int64_t device_bytes;    /* size of the device weight image (qlin_bind) */
  float alpha;             /* W8A8 migration strength (0 otherwise) */
  float outlier_frac;      /* SpQR outlier fraction (0 otherwise) */
} qlin_layer_info;

/* Host pointers into the handle's canonical arrays (valid until qlin_destroy).  Fields a
 * format does not use are NULL.  Layouts:
 *  W4G128: codes uint32 [N][K/8] (nibble i of word j = k 8j+i), scale, zero fp16 [N][K/128].
 *  SPQR:   codes3 uint8 [N][3K/8] LSB-first 3-bit stream (code k at bits 3k..3k+2),
 *          qs3, qz3 uint8 [N][3(K/16)/8] same stream form, stats fp16 [N][K/256][4] =
 *          (ss, zs, sz, zz), rowptr int32 [N+1], col int16 [nnz], val fp16 [nnz].
 *  W8A8:   qw int8 [N][K], sw fp32 [N], s fp32 [K], s_inv fp32 [K].
 *  W4G128 act-order (qlin_pack_w4g128_gptq with act_order): perm int32 [K], a permutation of
 *          0..K-1; the codes, scales and zeros are those of the layer W[:, perm] (column j is
 *          input channel perm[j]) and the forward multiplies by X[:, perm].  NULL otherwise.
 * fp16 values are passed as uint16_t bit patterns. */
typedef struct {
  const uint32_t* codes;
  const uint16_t* scale;
  const uint16_t* zero;
  const uint8_t* codes3;
  const uint8_t* qs3;
  const uint8_t* qz3;
  const uint16_t* stats;
  const int32_t* rowptr;
  const int16_t* col;
  const uint16_t* val;
  const int8_t* qw;
  const float* sw;
  const float* s;
  const float* s_inv;
  const int32_t* perm;
} qlin_canonical;

/* ---- checkpoint load (host) --------------------------------------------------------- */

/* A handle from canonical arrays in the layout qlin_export describes (a saved checkpoint):
 * the GPTQ page ("Makale Bülteni — GPTQ", open-source paragraphs) and the SmoothQuant page
 * ("Ticari Etki") describe inference engines loading already-quantized checkpoints; this is
 * that load, with no quantization -- the device image is built exactly as the packer of the
 * same format builds it, so forwards match the exporting handle bit for bit.
 * format: QLIN_FMT_*.  in: host pointers to the format's arrays (the others are ignored),
 * read only, not retained, sized as qlin_export documents (SpQR: nnz = rowptr[N]; col and val
 * may be NULL when nnz == 0).  Checked: shapes as for the packers; W4 scales positive finite,
 * zeros integers 0..15; SpQR stats finite with integer zs, zz in 0..7, rowptr starting at 0 and
 * non-decreasing with at most K entries per row, columns strictly ascending in [0, K), values
 * finite; W4 perm (optional) a permutation of 0..K-1; W8 qw >= -127, sw, s, s_inv positive
 * finite.  Anything else: INVALID_ARG.  The
 * info fields alpha (W8A8) and outlier_frac (SpQR: nnz / (N K)) are informational. */
qlin_status qlin_import(int format, int N, int K, const qlin_canonical* in, qlin_handle* out);

/* ---- packing (offline, host) ------------------------------------------------------ */

/* W4 g128, round-to-nearest asymmetric per (row, 128-group) (GPTQ page, see above).
 * W: host fp32 [N][K], read only, not retained.  K % 128 == 0, N >= 1, W finite.
 * Returns INVALID_ARG on bad shapes/values (a group whose scale overflows fp16 included). */
qlin_status qlin_pack_w4g128(const float* W, int N, int K, qlin_handle* out);

/* W4 g128 with GPTQ error compensation (GPTQ page, "Makale Bülteni — GPTQ" intro and
 * "İddia ve Gerçeklik: GPTQ": inverse Hessian from the covariance of the layer inputs,
 * stabilised by a Cholesky decomposition; columns quantized in order, each column's rounding
 * error spread at once over the columns not yet quantized).  Same handle, layout and kernels
 * as qlin_pack_w4g128.  Steps: H = Xcal^T Xcal (fp64); an always-zero input column gets
 * H_kk = 1 and zero weights; H += damp * mean(diag H) * I; U = upper Cholesky factor of H^-1;
 * at the first column of each 128-group the group's scale/zero are round-to-nearest over the
 * group's current weights (fp32); column k gets the round-to-nearest code with them, and
 * every later weight of the row moves by -e * U_kj, e = (w_k - w_hat_k) / U_kk (fp64).
 * With H = I the result equals qlin_pack_w4g128's bit for bit.
 * act_order != 0 (same page, last paragraph: columns ordered by activation size, groups then
 * irregular in the original order): the columns are taken by decreasing diag(H) (an
 * always-zero input counted as 1, ties to the smaller index) and W[:, perm] is quantized as
 * above under H[perm][perm]; the handle keeps perm (exported and imported with the codes),
 * and the forward reads X in the permuted order: one token with K <= 8192 is gathered by the
 * single-token kernel while it stages x, any other forward first gathers X[:, perm] into the
 * workspace (one more kernel launch; M <= the workspace's max_M) -- the run-time price the
 * page mentions.
 * W: host fp32 [N][K]; Xcal: host fp32 [S][K] calibration inputs (row-major); both read only,
 * not retained.  K % 128 == 0, K <= 8192 (H and its factors are K x K fp64 on the host),
 * S >= 1, damp > 0 (0.01 is the usual value), W and Xcal finite.  Returns INVALID_ARG on bad
 * shapes/values or if H + damping is not positive definite; the work is O(K^3 + N K^2). */
qlin_status qlin_pack_w4g128_gptq(const float* W, int N, int K, const float* Xcal, int S, double damp,
                                  int act_order, qlin_handle* out);

/* SpQR 3-bit g16 bi-level + fp16 CSR outliers (SpQR page, see above).  The outliers are
 * the floor(f*N*K) largest |w| (ties: smaller linear index), standing in for the page's
 * Hessian-sensitivity choice.  K % 256 == 0, K <= 32768 (int16 columns), 0 <= f < 1. */
qlin_status qlin_pack_spqr(const float* W, int N, int K, float outlier_frac, qlin_handle* out);

/* SmoothQuant W8 (SmoothQuant page, see above): s_k = max(ax_k,1e-5)^alpha /
 * max(aw_k,1e-5)^(1-alpha) (float64, rounded to fp32), aw_k = max_n |W[n][k]|;
 * W' = W diag(s); per-row int8 with sw_n = max|W'_n| / 127.
 * act_absmax: host fp32 [K], the calibration per-channel max |x|.  0 <= alpha <= 1. */
qlin_status qlin_pack_w8(const float* W, int N, int K, const float* act_absmax, float alpha,
                         qlin_handle* out);

/* ---- device residency ------------------------------------------------------------- */

/* Size in bytes of the device weight image that qlin_bind uploads. */
qlin_status qlin_device_bytes(qlin_handle h, size_t* weight_bytes);

/* Workspace a forward with up to max_M rows needs (partial sums of split output rows,
 * their arrival counters, the device status word; W8A8: the activation codes and scales;
 * act-order W4: X in the permuted channel order). */
qlin_status qlin_workspace_bytes(qlin_handle h, int max_M, size_t* bytes);

/* Copies the device image into caller-owned device memory dev_weights (>= weight_bytes,
 * 256-byte aligned) with cudaMemcpyAsync on `stream`.  The handle keeps the host image
 * alive, so the caller need not wait before returning. */
qlin_status qlin_bind(qlin_handle h, void* dev_weights, size_t bytes, qlin_stream stream);

/* Points the handle at device memory that already holds its image (for example a
 * device-to-device copy of a bound image), without copying anything.  Lets one packed
 * layer run from several resident copies.  Same size/alignment rules as qlin_bind. */
qlin_status qlin_attach(qlin_handle h, void* dev_weights, size_t bytes);

/* Hands the handle a caller-owned device workspace (256-byte aligned) and clears its
 * counters and status word on `stream`.  max_M is the largest M later forwards will use. */
qlin_status qlin_set_workspace(qlin_handle h, void* dev_ws, size_t bytes, int max_M,
                               qlin_stream stream);

/* ---- forward ---------------------------------------------------------------------- */

/* Y = X . W_hat^T.  X: device bf16 [M][K], Y: device bf16 [M][N], both 16-byte aligned.
 * Asynchronous on `stream`; returns launch errors only.  M == 0 is a no-op.  Decode
 * (1 <= M <= 16) runs the fused dequant GEMV kernels; larger M runs the tensor-core path.
 * W8A8 and act-order W4 handles keep per-token data in the workspace, so for them M must
 * not exceed the workspace's max_M (QLIN_ERR_WORKSPACE otherwise). */
qlin_status qlin_forward(qlin_handle h, const void* X, void* Y, int M, qlin_stream stream);

/* The SpQR decode forward (format SPQR, 1 <= M <= 16) without any workspace: for callers
 * that are given only X and Y and may not allocate device memory -- a layer inside an engine
 * that reserves all device memory for its own pools and hands plugins no workspace, or a
 * service that forbids device allocation once it is serving.  The pages have no counterpart;
 * this is a deployment form of qlin_forward: the same kernels, and the same outputs bit for
 * bit.
 * The scratch (partial sums of split row groups, their counters or tags, a status word) is a
 * fixed array of about 8 MB inside the library.  It is taken on a device when the library's
 * device module is loaded there -- under CUDA's lazy module loading, at the first qlin_bind
 * or qlin_attach of a SpQR handle on that device, which look up its address for that reason
 * (or else at the first call of this function) -- and held until the process exits.  Make
 * that first bind or call before any stream capture and before the device's memory is
 * reserved for other uses.
 * Limits: layers of at most 162,560 units of 64 rows x 256 columns (ceil(N / 64) * K / 256), at
 * most 524,288 rows, on devices of at most 160 SMs; beyond them the call returns
 * QLIN_ERR_WORKSPACE.  Each call clears the counters it uses; the array is shared by every
 * call, so calls whose kernels overlap on the GPU (other streams, other threads) race and
 * must be serialized by the caller.  A device-side wait that gives up is recorded in the
 * array's status word and reported by qlin_poll_static_status.  Allocates nothing: no
 * cudaMalloc, cudaFree or allocating library call. */
qlin_status qlin_forward_spqr_static(qlin_handle h, const void* X, void* Y, int M, qlin_stream stream);

/* Status of the qlin_forward_spqr_static calls on the current device since the last poll:
 * waits for `stream`, then reads and clears the fixed array's status word.  QLIN_OK, or
 * QLIN_ERR_TIMEOUT if a device-side wait gave up (the outputs of that call are then
 * incomplete).  No counterpart on the pages. */
qlin_status qlin_poll_static_status(qlin_stream stream);

/* End-to-end form: copies X from host memory (X_host, pinned for full speed) into X_dev,
 * runs qlin_forward, copies Y_dev back into Y_host and waits for the stream.  On a created
 * stream the three steps are captured once into a CUDA graph per (X_host, Y_host, X_dev, Y_dev,
 * bound weights, M, stream) and replayed on later calls with the same arguments (up to 64 kept
 * per handle, least recently used dropped; qlin_set_workspace drops them all); on the legacy
 * default stream, or while the stream is being captured by the caller, they are enqueued one by
 * one.  The host buffers are read and written when the step runs, as with plain copies. */
qlin_status qlin_forward_host(qlin_handle h, const void* X_host, void* Y_host, void* X_dev,
                              void* Y_dev, int M, qlin_stream stream);

/* W8A8 only: the per-token activation quantization step alone (int8 codes and fp32
 * scales of X diag(s)^-1).  qx: device int8 [M][K], sx: device fp32 [M]. */
qlin_status qlin_act_quant(qlin_handle h, const void* X, int8_t* qx, float* sx, int M,
                           qlin_stream stream);

/* W8A8 only: the exact int32 accumulators acc[m][n] = sum_k qx[m][k] * qw[n][k] of a
 * forward, instead of Y.  acc: device int32 [M][N]. */
qlin_status qlin_forward_acc(qlin_handle h, const void* X, int32_t* acc, int M,
                             qlin_stream stream);

/* Writes the dequantized fp32 weights W_hat [N][K] decoded from the bound device image
 * (W4G128, SPQR), or the int8 codes qw [N][K] (W8A8, out viewed as int8).  Checks that
 * the device layout decodes to exactly the canonical arrays.  Act-order W4: the columns come
 * in the codes' (permuted) order, column j being input channel perm[j]. */
qlin_status qlin_dequant_device(qlin_handle h, void* out, qlin_stream stream);

/* Waits for `stream`, then reads and clears the device status word: QLIN_OK or
 * QLIN_ERR_TIMEOUT if a device-side wait gave up since the last poll. */
qlin_status qlin_poll_status(qlin_handle h, qlin_stream stream);

/* ---- inspection ------------------------------------------------------------------- */

qlin_status qlin_export(qlin_handle h, qlin_canonical* out);
qlin_status qlin_info(qlin_handle h, qlin_layer_info* out);
void qlin_destroy(qlin_handle h);
const char* qlin_status_string(qlin_status s);

/* Number of SMs the kernels size their grids for (queried on the current device). */
int qlin_sm_count(void);

/* Test hook for device-side wait limits: launches one block that waits on an mbarrier
 * nothing ever arrives on, with a wall-time limit of limit_us microseconds (1 .. 10^7); the
 * block then records QLIN_ERR_TIMEOUT in status (device int32) and exits cleanly.  Every
 * wait inside the library's kernels has the same kind of limit (2 s). */
qlin_status qlin_debug_wait_timeout(int32_t* status, int limit_us, qlin_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_H_ */

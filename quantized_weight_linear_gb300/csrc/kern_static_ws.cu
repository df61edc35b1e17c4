// SpQR decode forward that allocates nothing: its scratch lives in a fixed array compiled
// into the library instead of a caller-provided workspace.
//
// Who needs it: code that is handed only its input and output buffers and may not call
// cudaMalloc -- a layer plugged into an inference engine that reserves the whole device
// memory up front for its own pools and gives plugins no workspace, or a service that forbids
// any device allocation after start-up because an allocation can stall or fail while
// requests are in flight.  qlin_forward needs a workspace (split-row partial sums, their
// arrival counters or tags, and the status word); this entry point takes that scratch from
// `g_spqr_static_scratch` below.
//
// Limits of the fixed array: partial-sum slots for at most kStaticMaxGrid CTAs or workers,
// which holds every layer of at most 162,560 units of 64 rows x 256 columns (RG x K / 256) on a
// device of at most 160 SMs, and kStaticMaxRowGroups row groups of 64 output rows
// (N <= 524288); larger requests return QLIN_ERR_WORKSPACE.  The array (about 8 MB) is part of
// this library's device module: it is taken on a device when the module is loaded there --
// with lazy module loading, at the first address lookup, which qlin_bind / qlin_attach of a
// SpQR handle make (qlin_static_scratch_prepare) -- and held until the process exits.
#include <mutex>

#include "../../include/qlin.h"
#include "kern_common.cuh"

namespace qlin {
namespace {

constexpr int kStaticMaxGrid = 640;
constexpr int kStaticMaxRowGroups = 8192;
constexpr size_t kStaticPartialsOff = 256;
constexpr size_t kStaticCountersOff = kStaticPartialsOff + (size_t)kStaticMaxGrid * 2 * kRowGroup * 16 * 4;
constexpr size_t kStaticTaggedOff = kStaticCountersOff + (size_t)kStaticMaxRowGroups * 4;
constexpr size_t kStaticScratchBytes = kStaticTaggedOff + (size_t)kStaticMaxGrid * 2 * kRowGroup * 4 * 8;
constexpr int kMaxDevices = 64;

// [0, 256): status word; then partial slots, arrival counters, tagged words.  Zero at load.
static __device__ __align__(256) unsigned char g_spqr_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_dev_ptr[kMaxDevices];
uint32_t g_tag[kMaxDevices];  // tag of the last call on each device

// Device address of the scratch array on the current device, looked up once per device
// (cudaGetSymbolAddress with that device current, which also loads the module there), then
// cached.  Caller holds g_mu.
qlin_status scratch_address_locked(int dev, uint8_t** out) {
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_spqr_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return QLIN_ERR_CUDA;
    }
    g_dev_ptr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_dev_ptr[dev]);
  return QLIN_OK;
}

qlin_status current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) {
    cudaGetLastError();
    return QLIN_ERR_CUDA;
  }
  return QLIN_OK;
}

qlin_status scratch_on_current_device(uint8_t** out, int* sms, uint32_t* tag) {
  int dev = 0;
  if (qlin_status s = current_device(&dev)) return s;
  std::lock_guard<std::mutex> lock(g_mu);
  if (qlin_status s = scratch_address_locked(dev, out)) return s;
  if (++g_tag[dev] == 0u) g_tag[dev] = 1u;  // 0 marks a word as not written
  *tag = g_tag[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return QLIN_ERR_CUDA;
  *sms = n;
  return QLIN_OK;
}

}  // namespace

// Loads the scratch array on the current device (see the file comment); called by qlin_bind
// and qlin_attach for SpQR handles, so that the array is in place before a caller reserves
// the device's memory for other uses.
int qlin_static_scratch_prepare() {
  int dev = 0;
  if (qlin_status s = current_device(&dev)) return s;
  std::lock_guard<std::mutex> lock(g_mu);
  uint8_t* p = nullptr;
  return scratch_address_locked(dev, &p);
}

}  // namespace qlin

using namespace qlin;

extern "C" qlin_status qlin_forward_spqr_static(qlin_handle h, const void* X, void* Y, int M, qlin_stream stream) {
  SpqrView v;
  if (!h || M < 0 || M > 16) return QLIN_ERR_INVALID_ARG;
  const int st = qlin_spqr_view_of(h, &v);
  if (st != QLIN_OK) return (qlin_status)st;
  if (M == 0) return QLIN_OK;
  if (!X || !Y || ((uintptr_t)X & 15u) || ((uintptr_t)Y & 15u)) return QLIN_ERR_INVALID_ARG;
  uint8_t* scratch = nullptr;
  int sms = 0;
  uint32_t tag = 0;
  qlin_status s = scratch_on_current_device(&scratch, &sms, &tag);
  if (s != QLIN_OK) return s;
  const int slots = M == 1 ? gemv1_slots((int64_t)v.RG * v.S, sms, true) : spqr_decode_grid(v, M, sms);
  if (slots > kStaticMaxGrid || v.RG > kStaticMaxRowGroups) return QLIN_ERR_WORKSPACE;
  // the array keeps the previous call's contents: clear the arrival counters (plain partial
  // slots are always written before they are read, and tagged words carry a tag of this
  // call's own); the status word is kept until qlin_poll_static_status reads it
  cudaStream_t cs = (cudaStream_t)stream;
  if (cudaMemsetAsync(scratch + kStaticCountersOff, 0, (size_t)v.RG * 4, cs) != cudaSuccess) return QLIN_ERR_CUDA;
  Workspace ws{};
  ws.status = reinterpret_cast<int32_t*>(scratch);
  ws.partials = reinterpret_cast<float*>(scratch + kStaticPartialsOff);
  ws.counters = reinterpret_cast<uint32_t*>(scratch + kStaticCountersOff);
  ws.tagged = reinterpret_cast<uint64_t*>(scratch + kStaticTaggedOff);
  ws.tag = tag;
  ws.qx = nullptr;
  ws.sx = nullptr;
  ws.grid = kStaticMaxGrid;
  ws.sms = sms;
  const int e = launch_spqr_decode(v, (const uint16_t*)X, (uint16_t*)Y, M, ws, 0, stream);
  return e ? QLIN_ERR_CUDA : QLIN_OK;
}

extern "C" qlin_status qlin_poll_static_status(qlin_stream stream) {
  uint8_t* scratch = nullptr;
  int dev = 0;
  if (qlin_status s = current_device(&dev)) return s;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (qlin_status s = scratch_address_locked(dev, &scratch)) return s;
  }
  cudaStream_t cs = (cudaStream_t)stream;
  int32_t status = 0;
  if (cudaMemcpyAsync(&status, scratch, sizeof(status), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
      cudaMemsetAsync(scratch, 0, sizeof(status), cs) != cudaSuccess || cudaStreamSynchronize(cs) != cudaSuccess)
    return QLIN_ERR_CUDA;
  return status == kStatusOk ? QLIN_OK : QLIN_ERR_TIMEOUT;
}

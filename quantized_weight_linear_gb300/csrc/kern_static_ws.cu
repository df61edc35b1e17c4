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
// Limits of the fixed array: at most kStaticMaxGrid CTAs (4 per SM on up to 160 SMs) and
// kStaticMaxRowGroups row groups of 64 output rows (N <= 524288); larger requests return
// QLIN_ERR_WORKSPACE.  Every GPU that loads the library holds the array (about 8 MB) until
// the process exits.
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

static __device__ __align__(256) unsigned char g_spqr_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_dev_ptr[kMaxDevices];
uint32_t g_tag[kMaxDevices];  // tag of the last call on each device

// Device address of the scratch array on the current device; looked up once per device
// (cudaGetSymbolAddress with that device current), then cached.
qlin_status scratch_on_current_device(uint8_t** out, int* sms, uint32_t* tag) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QLIN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_spqr_static_scratch) != cudaSuccess || !p) return QLIN_ERR_CUDA;
    g_dev_ptr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_dev_ptr[dev]);
  if (++g_tag[dev] == 0u) g_tag[dev] = 1u;  // 0 marks a word as not written
  *tag = g_tag[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return QLIN_ERR_CUDA;
  *sms = n;
  return QLIN_OK;
}

}  // namespace
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
  const int grid = spqr_decode_grid(v, M, sms);
  if (grid > kStaticMaxGrid || v.RG > kStaticMaxRowGroups) return QLIN_ERR_WORKSPACE;
  // the array keeps the previous call's contents: clear the status word and the counters
  // (plain partial slots are always written before they are read, and tagged words carry a
  // tag of this call's own)
  cudaStream_t cs = (cudaStream_t)stream;
  if (cudaMemsetAsync(scratch, 0, 256, cs) != cudaSuccess) return QLIN_ERR_CUDA;
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
  const int e = launch_spqr_decode(v, (const uint16_t*)X, (uint16_t*)Y, M, ws, grid, stream);
  return e ? QLIN_ERR_CUDA : QLIN_OK;
}

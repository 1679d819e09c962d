// logprob_static_scratch.cu -- iso_selected_logprob_static_scratch: the
// selected-token logprob for callers that cannot allocate device memory.
//
// Who needs it: code that reaches this library through a plugin or callback
// interface that hands it only input and output pointers -- no allocator and
// no workspace argument -- and code that must not call cudaMalloc because the
// framework around it owns every byte of device memory (a serving engine's
// pre-reserved pool) or because cudaMalloc would synchronize the device in the
// middle of its hot loop.  Such callers cannot provide the workspace that
// iso_selected_logprob asks for.
//
// What it does: the scratch lives in one file-scope device array of fixed
// size (ISO_LOGPROB_STATIC_SCRATCH_BYTES).  The array exists on every GPU
// that loads this library, from load until process exit.  The entry point
// looks up the array's device address once per device (the first call made
// with that device current does it; make that first call before any stream
// capture), then runs exactly the kernels of iso_selected_logprob with the
// array as their workspace, so the results are bit-identical to that entry
// point's.  Nothing is allocated or freed.
//
// Sharing: every call on a device uses the same array and leaves its contents
// behind.  No byte of it needs to start at zero -- each entry the kernels read
// is first written by the same call -- but two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on the array and
// may return wrong values.  Serialize such calls on one stream.
#include <mutex>

#include "iso_internal.h"

static __device__ __align__(256) unsigned char g_iso_logprob_scratch[ISO_LOGPROB_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevicesScratch = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevicesScratch] = {};

// Host code may not use g_iso_logprob_scratch's name as a device address (on
// the host it is only a stand-in); ask the runtime for the real one.
iso_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesScratch) return ISO_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_iso_logprob_scratch) != cudaSuccess || p == nullptr) return ISO_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ISO_OK;
}

}  // namespace

extern "C" iso_status iso_selected_logprob_static_scratch(const iso_contract* c, const iso_bf16* h, const iso_bf16* W,
                                                          const int32_t* ids, float* out, int T, int H, int V,
                                                          iso_stream stream) {
  if (!c || T < 0 || H <= 0 || V <= 0) return ISO_ERR_INVALID_ARG;
  if (T == 0) return ISO_OK;
  const size_t need = iso_selected_logprob_min_workspace(c, T, V);
  if (need == 0 || need > static_cast<size_t>(ISO_LOGPROB_STATIC_SCRATCH_BYTES)) return ISO_ERR_WORKSPACE;
  void* scratch = nullptr;
  const iso_status st = scratch_for_current_device(&scratch);
  if (st != ISO_OK) return st;
  return iso_selected_logprob(c, h, W, ids, out, T, H, V, scratch, static_cast<size_t>(ISO_LOGPROB_STATIC_SCRATCH_BYTES),
                              stream);
}

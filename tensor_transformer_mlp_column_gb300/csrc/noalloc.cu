// noalloc.cu — a forward entry point that allocates no memory at all.
//
// Some callers cannot allocate device memory when they call this library:
// runtimes that reserve every byte of the GPU up front and hand it out only
// through their own pool, so a cudaMalloc (or a torch allocation) outside
// that pool is forbidden or fails; and loops that cannot afford the implicit
// device synchronisation that cudaMalloc/cudaFree bring. Such callers cannot
// size and pass the scratch buffer that tpmlp_forward needs. This entry point
// uses a fixed scratch array in device memory instead, reserved once per GPU
// when the library's device code is loaded and held until the process exits.
//
// The scratch array holds at most kScratchBytes (64 MiB); a call whose
// workspace (tpmlp_workspace_bytes of the same T, shards and mode) would be
// larger is refused with TPMLP_ERR_WORKSPACE before anything is enqueued.
// All calls on a GPU share the one array: two calls whose work overlaps on
// the GPU (different streams, or different host threads, without ordering
// between them) race on it and give wrong results. Nothing in the array has
// to start at zero: every byte a call reads was written earlier by that same
// call. The array keeps whatever the last call left in it.
#include "tpmlp.h"

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per GPU

// The scratch itself. In host code this name only stands for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device. Looked up once
// per device, the first time this entry point runs there.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tpmlp::set_error(TPMLP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return tpmlp::set_error(TPMLP_ERR_DEVICE, "device index %d unsupported", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return tpmlp::set_error(TPMLP_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                              cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TPMLP_OK;
}

}  // namespace

extern "C" int tpmlp_forward_noalloc(const void* X, int64_t T, const tpmlp_shards* shards, void* Y, tpmlp_mode mode,
                                     tpmlp_stream_t stream) {
  if (!shards) return tpmlp::set_error(TPMLP_ERR_ARG, "shards handle is NULL");
  if (T < 1) return tpmlp::set_error(TPMLP_ERR_ARG, "T = %lld must be >= 1", static_cast<long long>(T));
  if (mode != TPMLP_FAITHFUL && mode != TPMLP_FUSED) return tpmlp::set_error(TPMLP_ERR_ARG, "unknown mode %d", int(mode));
  const size_t need = tpmlp_workspace_bytes(T, shards, mode, 0);
  if (need == 0 || need > kScratchBytes)
    return tpmlp::set_error(TPMLP_ERR_WORKSPACE,
                            "this call needs %zu bytes of scratch but the static scratch holds %zu bytes (64 MiB); "
                            "use fewer tokens per call, the fused mode, or tpmlp_forward with a workspace",
                            need, kScratchBytes);
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  return tpmlp_forward(X, T, shards, Y, mode, scratch, kScratchBytes, stream);
}

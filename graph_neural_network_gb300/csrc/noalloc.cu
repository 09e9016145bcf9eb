// Forward pass for callers that cannot allocate device memory.
//
// Same kernels as gat_agg_forward; the only difference is where the hub
// partial states live: in a fixed-size array that belongs to this library
// (one per GPU that loads it, held until the process exits) instead of a
// workspace the caller allocates.
#include <cuda.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;

// The array's device address on each device, with the id of the context it
// was looked up in: a device reset (or a released and re-created primary
// context) loads the module again at a new address, so a cached address is
// used only while the current context is the one it came from.
struct ScratchAddr {
  unsigned long long ctx_id;
  void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the calling thread's current context, 0 when there is none or the
// driver cannot say (the address is then looked up again).
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
      get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    resolved = true;
  }
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch on `dev` (which must be current).  In
// host code the symbol's name is only a host-side stand-in, so the address
// is looked up with cudaGetSymbolAddress the first time a context of the
// device calls, and cached for that context.
cudaError_t scratch_on_device(int dev, void** addr) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  ScratchAddr& c = g_scratch_addr[dev];
  const unsigned long long id = current_ctx_id();
  if (!c.addr || id == 0 || c.ctx_id != id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    c.addr = p;
    c.ctx_id = current_ctx_id();  // the lookup may have created the context
  }
  *addr = c.addr;
  return cudaSuccess;
}

bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" size_t gat_agg_forward_noalloc_capacity(void) { return kNoAllocScratchBytes; }

extern "C" gnn_status gat_agg_forward_noalloc(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                              const void* h, const float* a_src,
                                              const float* a_dst, float slope, void* out,
                                              float* lse, void* stream) {
  if (!g || H < 1 || D < 1 || (dtype != GNN_F32 && dtype != GNN_BF16)) return GNN_ERR_INVALID_ARG;
  gnn::Shape s;
  if (!gnn::make_shape(H, D, dtype, &s)) return GNN_ERR_UNSUPPORTED;
  if (g->n == 0) return GNN_OK;
  if (!h || !a_src || !a_dst || !out || !lse) return GNN_ERR_INVALID_ARG;
  if (!aligned_to(h, 16) || !aligned_to(out, 16) || !aligned_to(a_src, 16) ||
      !aligned_to(a_dst, 16) || !aligned_to(lse, 4))
    return GNN_ERR_INVALID_ARG;
  const gnn::WsLayout L = gnn::ws_layout(g, s);
  if (L.fwd_total > kNoAllocScratchBytes) return GNN_ERR_WORKSPACE_TOO_SMALL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GNN_ERR_CUDA;
  if (dev != g->device || dev < 0 || dev >= kMaxDevices) return GNN_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (scratch_on_device(dev, &ws) != cudaSuccess) return GNN_ERR_CUDA;
  const cudaError_t e =
      gnn::launch_forward(g, s, dtype, h, a_src, a_dst, slope, out, lse, static_cast<char*>(ws),
                          L, static_cast<cudaStream_t>(stream), nullptr);
  return e == cudaSuccess ? GNN_OK : GNN_ERR_CUDA;
}

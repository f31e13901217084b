// bf16_attn_bwd_static: the backward with its workspace in a fixed device array of this library
// instead of caller memory, so the call allocates nothing and needs no buffer from the caller.
// The array lives in its own translation unit: with lazily loaded modules its memory is taken only
// by processes that make this call.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "bsc.h"

namespace {

// 256 MiB: the backward at B=1, Hq=16, Hkv=4, S=32K needs 205 MB; larger calls are refused.
constexpr size_t kStaticWorkspaceBytes = size_t(256) << 20;
static __device__ __align__(256) uint8_t g_bwd_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};   // the array's address, per device (set up on the first call there)

}  // namespace

extern "C" size_t bf16_attn_bwd_static_capacity(void) { return kStaticWorkspaceBytes; }

extern "C" bsc_status bf16_attn_bwd_static(const bsc_attn_bwd_params* p, bsc_stream_t stream) {
  if (!p) return BSC_ERR_NULL;
  if (bf16_attn_bwd_workspace_bytes(p->B, p->S, p->Hq, p->Hkv) > kStaticWorkspaceBytes) return BSC_ERR_SHAPE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSC_ERR_CUDA;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      if (cudaGetSymbolAddress(&g_addr[dev], g_bwd_workspace) != cudaSuccess) {
        g_addr[dev] = nullptr;
        return BSC_ERR_CUDA;
      }
    }
    ws = g_addr[dev];
  }
  bsc_attn_bwd_params q = *p;
  q.workspace = static_cast<float*>(ws);
  q.workspace_bytes = kStaticWorkspaceBytes;
  return bf16_attn_bwd(&q, stream);
}

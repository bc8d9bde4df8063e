// Grouped-head decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: an engine whose
// own allocator has already reserved nearly all of HBM (a cudaMalloc would
// fail, or fragment its pool), a plug-in host that exposes no device
// allocator to the code it loads, or a latency-critical loop where the
// implicit synchronisation of cudaMalloc/cudaFree is not acceptable. For them
// gqa_decode_no_alloc runs the same split-KV kernels as gqa_decode, with the
// split partials kept in a fixed array in this library's device image instead
// of a caller workspace. Nothing here calls cudaMalloc, cudaFree or any
// allocating library routine.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its DECATTN_NO_ALLOC_SCRATCH_BYTES until the process exits.
// Host code only sees a host-side stand-in for its name, so its device
// address is looked up once per device with cudaGetSymbolAddress (on the
// first call made while that device is current) and passed to the kernels.
#include <cstdint>
#include <mutex>

#include "decattn.h"

namespace {

constexpr size_t kScratchBytes = DECATTN_NO_ALLOC_SCRATCH_BYTES;

// Split partials (fp32 O, then fp32 LSE) of the last call on this device.
__device__ __align__(256) unsigned char g_no_alloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_no_alloc_scratch on the current device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DECATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_no_alloc_scratch) != cudaSuccess || !ptr) return DECATTN_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return DECATTN_OK;
}

}  // namespace

extern "C" int gqa_decode_no_alloc(const decattn_bf16* q, const decattn_bf16* k, const decattn_bf16* v,
                                   decattn_kv kv, const int32_t* seqlens, int max_seqlen, int b, int s, int hq,
                                   int hkv, int d, float scale, decattn_bf16* out, float* lse,
                                   cudaStream_t stream) {
  // The split plan (and so the partials' size) is the one gqa_decode uses;
  // invalid shapes give 0 here and are refused by gqa_decode itself.
  const size_t need = gqa_decode_workspace_size(b, s, hq, hkv, d, max_seqlen);
  if (need > kScratchBytes) return DECATTN_ERR_WORKSPACE;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    if (int rc = scratch_address(&ws)) return rc;
    ws_bytes = kScratchBytes;
  }
  // Every partial the combine kernel reads is written first by the split
  // kernel of the same call, so nothing in the array has to start at zero.
  return gqa_decode(q, k, v, kv, seqlens, max_seqlen, b, s, hq, hkv, d, scale, out, lse, ws, ws_bytes, stream);
}

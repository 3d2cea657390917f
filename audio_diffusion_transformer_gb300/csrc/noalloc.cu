// noalloc.cu -- routed attention for callers that cannot allocate device memory.
//
// h3dit_routed_attention needs a caller-provided workspace for its scratch
// (tile means, tile scores, selected tiles, pooled branch, status word).  Some
// callers have no way to get one: code running inside a host framework that
// owns every device allocation, plugins loaded into a process whose allocator
// they may not call, or paths where a cudaMalloc would synchronise the device
// or break a memory budget fixed in advance.  This entry point serves them
// from a fixed scratch array compiled into the library instead.
//
// The array lives in every GPU that loads the library until the process
// exits.  All calls share it: each call overwrites what the previous one left
// there, and clears the status word it needs at zero before its kernels run.
// Two calls whose kernels overlap on the GPU (different streams, or different
// host threads) race on the array and give wrong results; serialise them.
#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device.  In host code the
// symbol is only a host-side stand-in, so the address is looked up on every call,
// with the caller's device current (a cheap call that stays valid if the context
// has been torn down and made again since the last one).
h3dit_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
    return H3DIT_ERR_CUDA;
  *out = p;
  return H3DIT_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" h3dit_status h3dit_routed_attention_static(
    const h3dit_shape* shape, const void* q, const void* k, const void* v,
    const void* gate_or_null, void* out, float* pooled_out_or_null, int* topk_idx_out_or_null,
    float* tile_scores_out_or_null, void* stream) {
  // every argument check comes before the first CUDA call
  if (!shape) return H3DIT_ERR_ARG;
  h3dit_shape s = *shape;
  s.hidden = 0;     // size the attention-only scratch, as h3dit_routed_attention does
  s.mlp_width = 0;
  const size_t need = h3dit_workspace_bytes(&s);
  if (need == 0) return H3DIT_ERR_SHAPE;
  if (need > kStaticScratchBytes) return H3DIT_ERR_WORKSPACE;  // beyond the fixed scratch
  if (!q || !k || !v || !out) return H3DIT_ERR_ARG;
  const void* ptrs[] = {q, k, v, out, gate_or_null, pooled_out_or_null, topk_idx_out_or_null,
                        tile_scores_out_or_null};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return H3DIT_ERR_ALIGN;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return H3DIT_ERR_CUDA;
  if (major != 10) return H3DIT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const h3dit_status st = scratch_address(&scratch);
  if (st != H3DIT_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // the status word at the start of the scratch must read zero when the kernels start
  if (cudaMemsetAsync(scratch, 0, 256, cs) != cudaSuccess) return H3DIT_ERR_CUDA;
  return h3dit_routed_attention(&s, q, k, v, gate_or_null, out, pooled_out_or_null,
                                topk_idx_out_or_null, tile_scores_out_or_null, scratch,
                                kStaticScratchBytes, stream);
}

extern "C" h3dit_status h3dit_routed_attention_static_status(void* stream) {
  void* scratch = nullptr;
  const h3dit_status st = scratch_address(&scratch);
  if (st != H3DIT_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return H3DIT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return H3DIT_ERR_CUDA;
  if (v != 0 && cudaMemset(scratch, 0, sizeof(int)) != cudaSuccess) return H3DIT_ERR_CUDA;
  return static_cast<h3dit_status>(v);
}

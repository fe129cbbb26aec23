// msa_proxy_select_noalloc: proxy scoring and block selection for callers that
// cannot hand the library any device memory of its own.
//
// msa_proxy_select needs a small caller-owned workspace: the per-document
// block prefix (num_docs + 2 int32) that the metadata kernel writes and the
// selection kernel reads.  Here that scratch lives in a file-scope device
// array instead, so the call allocates nothing.  The array is part of the
// library image: every GPU that loads the library holds its 64 KB until the
// process exits.
#include <mutex>

#include "msa_internal.cuh"

namespace msa {
namespace {

// Largest batch, in documents, this entry point accepts.
constexpr int kNoAllocMaxDocs = 16382;

// The scratch: cu_blocks[0..num_docs] plus the well-formed flag at
// [num_docs + 1].  Every entry a call reads is written earlier in the same
// call, so nothing needs clearing between calls.
static __device__ __align__(256) int32_t g_noalloc_cu_blocks[kNoAllocMaxDocs + 2];

constexpr int kMaxDevicesNA = 64;
int32_t* g_noalloc_ptr[kMaxDevicesNA] = {};
std::mutex g_noalloc_mu;

// In host code the array's name is only a host-side stand-in; its device
// address is resolved once per device, with that device current.
cudaError_t noalloc_scratch(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesNA) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_cu_blocks);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" msa_status msa_proxy_select_noalloc(const msa_params* p, const int32_t* cu_seqlens,
                                               const uint16_t* q_p, const uint16_t* k_p,
                                               int32_t* sel_idx, float* sel_score,
                                               uint8_t* sel_arg, float* plse, uint8_t* tie,
                                               msa_stream_t stream) {
  Shape s;
  const msa_status st = check_params(p, &s);
  if (st != MSA_OK) return st;
  if (s.ndoc > kNoAllocMaxDocs) return MSA_ERR_WORKSPACE;  // beyond the static scratch
  if (s.T == 0) return MSA_OK;
  if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return MSA_ERR_INVALID_ARG;
  for (const void* ptr : {(const void*)q_p, (const void*)k_p, (const void*)sel_idx,
                          (const void*)sel_score, (const void*)sel_arg, (const void*)plse,
                          (const void*)tie})
    if (!ptr || !aligned16(ptr)) return MSA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int32_t* cu_blocks = nullptr;
  if (status_ptr(&status) != cudaSuccess) return MSA_ERR_CUDA;
  if (noalloc_scratch(&cu_blocks) != cudaSuccess) return MSA_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (launch_meta(s, cu_seqlens, cu_blocks, status, cs) != cudaSuccess) return MSA_ERR_CUDA;
  // no workspace for the block lists: the selector finds every argmax itself
  if (launch_select(s, cu_seqlens, cu_blocks, q_p, k_p, sel_idx, sel_score, sel_arg, plse, tie,
                    /*with_arg=*/true, status, cs) != cudaSuccess)
    return MSA_ERR_CUDA;
  add_launches(2);
  return MSA_OK;
}

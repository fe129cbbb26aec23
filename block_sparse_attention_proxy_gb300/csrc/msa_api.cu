// C ABI of libmsa: argument checks, workspace layout and launch sequencing.
// See include/msa.h for the contract of every entry point.
#include <atomic>
#include <cmath>
#include <mutex>

#include <cstdlib>

#include "msa_internal.cuh"

namespace msa {

// Device status word: first error recorded by any kernel of this library.
__device__ unsigned int g_msa_status = 0;

namespace {
constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

}  // namespace

// Address of this device's status word (resolved once per device).
cudaError_t status_ptr(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_msa_status);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

std::atomic<uint64_t> g_launches{0};
cudaEvent_t g_prof_start[4] = {}, g_prof_stop[4] = {};

}  // namespace

void add_launches(uint64_t n) { g_launches += n; }

namespace {

// Records the profiling event of kernel `which` (if one is set) on `st`.
cudaError_t prof_mark(int which, bool start, cudaStream_t st) {
  cudaEvent_t e = start ? g_prof_start[which] : g_prof_stop[which];
  return e ? cudaEventRecord(e, st) : cudaSuccess;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

msa_status check_params(const msa_params* p, Shape* s) {
  if (!p) return MSA_ERR_INVALID_ARG;
  if ((p->flags & ~(MSA_FLAG_REUSE_REGROUP | MSA_FLAG_TEST_STALL_SELECT)) != 0)
    return MSA_ERR_INVALID_ARG;
  if (p->total_tokens < 0 || p->num_docs < 1 || p->max_seqlen < 0) return MSA_ERR_INVALID_ARG;
  if (p->total_tokens > 0 && (p->max_seqlen < 1 || p->max_seqlen > p->total_tokens))
    return MSA_ERR_INVALID_ARG;
  if (p->hq <= 0 || p->hkv <= 0 || p->hq % p->hkv != 0) return MSA_ERR_INVALID_ARG;
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.f)) return MSA_ERR_INVALID_ARG;
  if (!(std::isfinite(p->proxy_scale) && p->proxy_scale > 0.f)) return MSA_ERR_INVALID_ARG;
  if (!std::isfinite(p->kl_weight)) return MSA_ERR_INVALID_ARG;
  const int G = p->hq / p->hkv;
  if (p->total_tokens >= kMaxTokens) return MSA_ERR_UNSUPPORTED;
  if (p->d != 64 && p->d != 128) return MSA_ERR_UNSUPPORTED;
  if (p->dp != 32 && p->dp != 64) return MSA_ERR_UNSUPPORTED;
  if (p->block != kBlock) return MSA_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MSA_ERR_UNSUPPORTED;
  if (p->hkv > 255 || p->hq > 255) return MSA_ERR_UNSUPPORTED;
  if (p->top_k < 1 || p->top_k > kMaxTopK) return MSA_ERR_UNSUPPORTED;
  if (p->window < 0 || p->window > p->top_k - 1 || p->dilation < 0) return MSA_ERR_INVALID_ARG;
  const long long nb = (long long)(p->total_tokens + kBlock - 1) / kBlock + p->num_docs;
  if (nb > kMaxBlocks) return MSA_ERR_UNSUPPORTED;
  s->T = p->total_tokens;
  s->ndoc = p->num_docs;
  s->max_seqlen = p->max_seqlen;
  s->hq = p->hq;
  s->hkv = p->hkv;
  s->G = G;
  s->d = p->d;
  s->dp = p->dp;
  s->K = p->top_k;
  s->window = p->window;
  // any spacing beyond the largest block index keeps no block; clamping keeps
  // window * dilation inside int
  s->dilation = p->dilation < 1 ? 1 : (p->dilation > kMaxBlocks ? kMaxBlocks : p->dilation);
  s->nb_bound = (int)nb;
  s->nchunks = (p->total_tokens + kChunkTokens - 1) / kChunkTokens;
  s->qc_blocks = kQChunkBlocks;
  if (const char* env = std::getenv("MSA_QUERY_CHUNK_BLOCKS")) {
    const long v = std::strtol(env, nullptr, 10);
    if (v > 0 && v < kQChunkBlocks) s->qc_blocks = (int)v;
  }
  s->nqchunks = (int)((nb + s->qc_blocks - 1) / s->qc_blocks);
  const long long qct = (long long)s->qc_blocks * kBlock;
  s->qc_tokens = p->total_tokens < qct ? p->total_tokens : (int)qct;
  s->softmax_scale = p->softmax_scale;
  s->proxy_scale = p->proxy_scale;
  s->kl_weight = p->kl_weight;
  s->test_stall_select = (p->flags & MSA_FLAG_TEST_STALL_SELECT) != 0;
  return MSA_OK;
}

namespace {

msa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

#define MSA_TRY(expr)                                 \
  do {                                                \
    const cudaError_t e__ = (expr);                   \
    if (e__ != cudaSuccess) return MSA_ERR_CUDA;      \
  } while (0)

}  // namespace

Workspace workspace_layout(const Shape& s, WsKind kind) {
  Workspace w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.cu_blocks = take((size_t)(s.ndoc + 2) * 4);  // + the well-formed flag
  // the block lists (regroup) form a prefix shared by all three calls
  {
    const size_t nbs = (size_t)s.nb_bound;
    w.chunk_range = take((size_t)2 * s.nchunks * 4);
    w.cnt = take((size_t)s.nchunks * s.hkv * nbs * 4);
    w.row_ptr = take(((size_t)s.hkv * nbs + 1) * 4);
    w.ent = take((size_t)s.T * s.hkv * (size_t)(s.K > 1 ? s.K - 1 : 1) * 4);
  }
  if (kind == kWsFwd) {
    // one query chunk: int16 partial rows, {lse, scale} per row
    w.o_part = take((size_t)s.qc_tokens * s.hq * s.K * s.d * 2);
    w.o_meta = take((size_t)s.qc_tokens * s.hq * s.K * 8);
  }
  if (kind == kWsBwd) {
    w.dsum = take((size_t)s.T * s.hq * 4);
    w.dq_part = take((size_t)s.qc_tokens * s.hq * s.K * s.d * 4);  // one query chunk, fp32
    w.kl_part = take((size_t)bwd_reduce_blocks(s) * 8 + 8);
    // one record per list entry (diagonal + gathered) of every (group, block),
    // plus one tile of padding read by the last tile's bulk copy
    w.rec = take(((size_t)s.T * s.hkv * s.K + 64) * bwd_rec_bytes(s.G));
  }
  w.total = off;
  return w;
}

cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                         uint64_t outer, uint32_t box_inner, uint32_t box_mid, uint32_t box_outer,
                         int swizzle_bytes) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  if (!g_encode) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {inner, mid, outer > 0 ? outer : 1};
  const cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  const cuuint32_t box[3] = {box_inner, box_mid, box_outer};
  const cuuint32_t es[3] = {1, 1, 1};
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  else if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  else if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r =
      g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_select_workspace_size(const msa_params* p) {
  Shape s;
  if (check_params(p, &s) != MSA_OK) return 0;
  return workspace_layout(s, kWsSelect).total;
}
size_t msa_fwd_workspace_size(const msa_params* p) {
  Shape s;
  if (check_params(p, &s) != MSA_OK) return 0;
  return workspace_layout(s, kWsFwd).total;
}
size_t msa_bwd_workspace_size(const msa_params* p) {
  Shape s;
  if (check_params(p, &s) != MSA_OK) return 0;
  return workspace_layout(s, kWsBwd).total;
}

msa_status msa_proxy_select(const msa_params* p, const int32_t* cu_seqlens, const uint16_t* q_p,
                            const uint16_t* k_p, int32_t* sel_idx, float* sel_score,
                            uint8_t* sel_arg, float* plse, uint8_t* tie, void* ws,
                            size_t ws_bytes, msa_stream_t stream) {
  Shape s;
  msa_status st = check_params(p, &s);
  if (st != MSA_OK) return st;
  if (s.T == 0) return MSA_OK;
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return MSA_ERR_INVALID_ARG;
  for (const void* ptr : {(const void*)q_p, (const void*)k_p, (const void*)sel_idx,
                          (const void*)sel_score, (const void*)sel_arg, (const void*)plse,
                          (const void*)tie})
    if (!ptr || !aligned(ptr, 16)) return MSA_ERR_INVALID_ARG;
  const Workspace w = workspace_layout(s, kWsSelect);
  if (!ws || !aligned(ws, 256)) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < w.total) return MSA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  MSA_TRY(status_ptr(&status));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* cu_blocks = reinterpret_cast<int32_t*>(base + w.cu_blocks);
  int32_t* chunk_range = reinterpret_cast<int32_t*>(base + w.chunk_range);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + w.cnt);
  int32_t* row_ptr = reinterpret_cast<int32_t*>(base + w.row_ptr);
  uint32_t* ent = reinterpret_cast<uint32_t*>(base + w.ent);
  MSA_TRY(launch_meta(s, cu_seqlens, cu_blocks, status, cs));
  MSA_TRY(prof_mark(1, true, cs));
  // block maxima, selection and the diagonal block's argmax
  MSA_TRY(launch_select(s, cu_seqlens, cu_blocks, q_p, k_p, sel_idx, sel_score, sel_arg, plse,
                        tie, /*with_arg=*/false, status, cs));
  MSA_TRY(prof_mark(1, false, cs));
  // the queries of every KV block, then the argmax of each chosen earlier block
  MSA_TRY(launch_regroup(s, cu_seqlens, cu_blocks, sel_idx, chunk_range, cnt, row_ptr, ent,
                         status, cs));
  MSA_TRY(launch_sel_arg(s, cu_seqlens, cu_blocks, row_ptr, ent, q_p, k_p, sel_arg, status, cs));
  g_launches += 7;
  return MSA_OK;
}

msa_status msa_fwd(const msa_params* p, const int32_t* cu_seqlens, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const int32_t* sel_idx, uint16_t* o,
                   uint16_t* o_res, float* lse, float* mass, void* ws, size_t ws_bytes,
                   msa_stream_t stream) {
  Shape s;
  msa_status st = check_params(p, &s);
  if (st != MSA_OK) return st;
  if (s.T == 0) return MSA_OK;
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return MSA_ERR_INVALID_ARG;
  for (const void* ptr : {(const void*)q, (const void*)k, (const void*)v, (const void*)sel_idx,
                          (const void*)o, (const void*)o_res, (const void*)lse, (const void*)mass})
    if (!ptr || !aligned(ptr, 16)) return MSA_ERR_INVALID_ARG;
  const Workspace w = workspace_layout(s, kWsFwd);
  if (!ws || !aligned(ws, 256)) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < w.total) return MSA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  MSA_TRY(status_ptr(&status));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* cu_blocks = reinterpret_cast<int32_t*>(base + w.cu_blocks);
  int32_t* chunk_range = reinterpret_cast<int32_t*>(base + w.chunk_range);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + w.cnt);
  int32_t* row_ptr = reinterpret_cast<int32_t*>(base + w.row_ptr);
  uint32_t* ent = reinterpret_cast<uint32_t*>(base + w.ent);
  int16_t* o_part = reinterpret_cast<int16_t*>(base + w.o_part);
  float2* o_meta = reinterpret_cast<float2*>(base + w.o_meta);
  const bool reuse = (p->flags & MSA_FLAG_REUSE_REGROUP) != 0;
  if (!reuse) {
    MSA_TRY(launch_meta(s, cu_seqlens, cu_blocks, status, cs));
    MSA_TRY(launch_regroup(s, cu_seqlens, cu_blocks, sel_idx, chunk_range, cnt, row_ptr, ent,
                           status, cs));
  }
  MSA_TRY(prof_mark(2, true, cs));
  // one pass per query chunk (a single pass, chunk = -1, when the batch fits one)
  const int nq = s.nqchunks;
  for (int c = 0; c < nq; ++c) {
    const int chunk = nq == 1 ? -1 : c;
    MSA_TRY(launch_fwd(s, cu_seqlens, cu_blocks, row_ptr, ent, q, k, v, o_part, o_meta, chunk,
                       status, cs));
    if (c == nq - 1) MSA_TRY(prof_mark(2, false, cs));
    MSA_TRY(launch_fwd_merge(s, cu_seqlens, cu_blocks, o_part, o_meta, o, o_res, lse, mass,
                             chunk, cs));
  }
  g_launches += (reuse ? 0 : 5) + 2 * nq;
  return MSA_OK;
}

msa_status msa_bwd(const msa_params* p, const int32_t* cu_seqlens, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const uint16_t* q_p, const uint16_t* k_p,
                   const uint16_t* o, const uint16_t* o_res, const float* lse, const float* mass,
                   const uint16_t* dO,
                   const int32_t* sel_idx, const float* sel_score, const uint8_t* sel_arg,
                   const float* plse, float* dq, float* dk, float* dv, float* dq_p, float* dk_p,
                   double* kl_loss, void* ws, size_t ws_bytes, msa_stream_t stream) {
  Shape s;
  msa_status st = check_params(p, &s);
  if (st != MSA_OK) return st;
  if (!kl_loss || !aligned(kl_loss, 8)) return MSA_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (s.T == 0) return cuda_status(cudaMemsetAsync(kl_loss, 0, sizeof(double), cs));
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return MSA_ERR_INVALID_ARG;
  for (const void* ptr :
       {(const void*)q, (const void*)k, (const void*)v, (const void*)q_p, (const void*)k_p,
        (const void*)o, (const void*)o_res, (const void*)lse, (const void*)mass, (const void*)dO,
        (const void*)sel_idx, (const void*)sel_score, (const void*)sel_arg, (const void*)plse,
        (const void*)dq, (const void*)dk, (const void*)dv, (const void*)dq_p, (const void*)dk_p})
    if (!ptr || !aligned(ptr, 16)) return MSA_ERR_INVALID_ARG;
  const Workspace w = workspace_layout(s, kWsBwd);
  if (!ws || !aligned(ws, 256)) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < w.total) return MSA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  MSA_TRY(status_ptr(&status));
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* cu_blocks = reinterpret_cast<int32_t*>(base + w.cu_blocks);
  int32_t* chunk_range = reinterpret_cast<int32_t*>(base + w.chunk_range);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(base + w.cnt);
  int32_t* row_ptr = reinterpret_cast<int32_t*>(base + w.row_ptr);
  uint32_t* ent = reinterpret_cast<uint32_t*>(base + w.ent);
  float* dsum = reinterpret_cast<float*>(base + w.dsum);
  float* dq_part = reinterpret_cast<float*>(base + w.dq_part);
  double* kl_part = reinterpret_cast<double*>(base + w.kl_part);
  const bool reuse = (p->flags & MSA_FLAG_REUSE_REGROUP) != 0;
  if (!reuse) {
    MSA_TRY(launch_meta(s, cu_seqlens, cu_blocks, status, cs));
    MSA_TRY(launch_regroup(s, cu_seqlens, cu_blocks, sel_idx, chunk_range, cnt, row_ptr, ent,
                           status, cs));
  }
  MSA_TRY(launch_bwd_pre(s, o, o_res, dO, dsum, cs));
  MSA_TRY(prof_mark(3, true, cs));
  // one pass per query chunk; with several, dK, dV and dk_p start from zero and
  // every pass adds its queries' share (chunk order, so the sum is deterministic)
  const int nq = s.nqchunks;
  if (nq > 1) {
    MSA_TRY(cudaMemsetAsync(dk, 0, (size_t)s.T * s.hkv * s.d * 4, cs));
    MSA_TRY(cudaMemsetAsync(dv, 0, (size_t)s.T * s.hkv * s.d * 4, cs));
    MSA_TRY(cudaMemsetAsync(dk_p, 0, (size_t)s.T * s.hkv * s.dp * 4, cs));
  }
  for (int c = 0; c < nq; ++c) {
    const int chunk = nq == 1 ? -1 : c;
    MSA_TRY(launch_bwd(s, cu_seqlens, cu_blocks, row_ptr, ent, base + w.rec, q, k, v, q_p, dO,
                       lse, dsum, mass, sel_score, sel_arg, plse, dq_part, dk, dv, dk_p, chunk,
                       status, cs));
    if (c == nq - 1) MSA_TRY(prof_mark(3, false, cs));
    MSA_TRY(launch_bwd_reduce(s, cu_seqlens, cu_blocks, dq_part, sel_idx, sel_score, sel_arg,
                              plse, mass, k_p, dq, dq_p, kl_part, kl_loss, chunk, c == nq - 1,
                              cs));
  }
  g_launches += (reuse ? 0 : 5) + 2 + 3 * nq;
  return MSA_OK;
}

uint64_t msa_launch_count(void) { return g_launches.load(); }

msa_status msa_set_profile_events(int which, msa_event_t start, msa_event_t stop) {
  if (which < 1 || which > 3) return MSA_ERR_INVALID_ARG;
  g_prof_start[which] = reinterpret_cast<cudaEvent_t>(start);
  g_prof_stop[which] = reinterpret_cast<cudaEvent_t>(stop);
  return MSA_OK;
}

static thread_local uint32_t t_last_status_word = 0;

uint32_t msa_last_status_word(void) { return t_last_status_word; }

msa_status msa_get_device_status(msa_stream_t stream) {
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return MSA_ERR_CUDA;
  unsigned* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return MSA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MSA_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return MSA_ERR_CUDA;
  t_last_status_word = v;
  return static_cast<msa_status>(v & 0xFFu);
}

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG: null/misaligned pointer or inconsistent sizes";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED: shape outside the supported set";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE: workspace smaller than required";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA: a CUDA call or kernel launch failed";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
    case MSA_ERR_DEVICE_CHECK: return "MSA_ERR_DEVICE_CHECK: malformed cu_seqlens or selection found on the device";
  }
  return "MSA_ERR_UNKNOWN";
}

}  // extern "C"

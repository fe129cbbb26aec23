// Declarations shared by the CUDA translation units of libmsa.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/msa.h"
#include "ptx.cuh"

namespace msa {

constexpr int kBlock = 128;        // KV block (tokens); also the query tile of the selector
constexpr int kMaxTopK = 16;       // slot index fits in 4 bits of a regroup entry
constexpr int kMaxBlocks = 49152;  // KV blocks per batch (regroup counters live in shared memory)
constexpr int kChunkTokens = 2048; // tokens per regroup chunk
constexpr int kMaxTokens = 1 << 27;
// Bounded waits give up after this many SM cycles (about 0.5-1 s at GB300 clocks).
constexpr long long kWaitCycles = 1000000000ll;

// Where a bounded wait gave up, stored above the status code in the status
// word: kernel id (4 bits), barrier index (8 bits), tile or block index (12 bits).
enum : uint32_t { kKerSelect = 1, kKerFwd = 2, kKerBwd = 3, kKerSelArg = 4 };
__host__ __device__ constexpr uint32_t wait_site(uint32_t kernel, uint32_t bar, int n) {
  return kernel | (bar << 4) | ((uint32_t)(n < 0 ? 0 : (n > 4095 ? 4095 : n)) << 12);
}

// ---------------------------------------------------------------------------
// device status word (first error wins)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(unsigned* status, unsigned code) {
  atomicCAS(status, 0u, code);
}

// Waits for phase `parity` of `bar`; gives up (records MSA_ERR_TIMEOUT and
// raises the CTA's abort flag) after kWaitCycles or as soon as another role of
// the CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* status, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      set_status(status, (uint32_t)MSA_ERR_TIMEOUT | (site << 8));
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag: lets this CTA's own asynchronous
// copies or MMAs land before the CTA exits or frees TMEM.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitCycles) {
  }
}
// Warp-uniform form: every lane waits, the result is the AND over the warp.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, unsigned* status,
                                              uint32_t site) {
  const bool ok = wait_bar(bar, parity, abort_flag, status, site);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// 16-bit fixed-point slot partials of the forward.  The normalised O of one
// (token, head, slot) is stored as int16 values q = rint(x * 32767 / m),
// m = max |x| over the row (one thread owns the row), with the fp32 scale
// m / 32767 beside it; the merge adds scale * q.  |x| <= m makes |q| <= 32767,
// and the error is at most m / 65534 per element: about 16 bits of the row's
// largest value, which the backward's D = rowsum(dO * O) needs (bf16, 8 bits,
// or fp16, 11 bits, partials are not enough).  The backward's dQ partials stay
// fp32: there one warp holds a row one element per lane, and the per-row
// maximum would take a cross-lane reduction per row.
// ---------------------------------------------------------------------------
constexpr float kQ16 = 32767.f;
// Magnitude bits of an fp32 value: for non-negative floats the integer order
// of the bits is the numeric order, so an integer max gives max |x| exactly.
__device__ __forceinline__ uint32_t abs_bits(uint32_t x) { return x & 0x7FFFFFFFu; }
// 32767 / m, or 0 for an all-zero row.
__device__ __forceinline__ float q16_factor(float m) { return m > 0.f ? __fdividef(kQ16, m) : 0.f; }
// a and b rounded to the nearest integer, packed as int16 with a in the low half.
__device__ __forceinline__ uint32_t pack_q16x2(float a, float b) {
  const int ia = __float2int_rn(a), ib = __float2int_rn(b);
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(d) : "r"(ia), "r"(ib));
  return d;
}
__device__ __forceinline__ float q16_lo(uint32_t x) { return (float)(int)(int16_t)(x & 0xFFFFu); }
__device__ __forceinline__ float q16_hi(uint32_t x) { return (float)((int)x >> 16); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Index of the document holding global token t (cu has ndoc+1 entries).
__device__ __forceinline__ int doc_of_token(const int32_t* cu, int ndoc, int t) {
  int lo = 0, hi = ndoc - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// Index of the document holding global block gb (cu_blocks has ndoc+1 entries).
__device__ __forceinline__ int doc_of_block(const int32_t* cu_blocks, int ndoc, int gb) {
  int lo = 0, hi = ndoc - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (cu_blocks[mid] <= gb) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bytes of one backward list-entry record for a group of G heads: a 16-byte
// header {token, slot, argmax offset, proxy coefficient} and G (LSE, D) pairs,
// padded to a multiple of 16 bytes.
__host__ __device__ constexpr int bwd_rec_bytes(int G) { return 16 + ((8 * G + 15) / 16) * 16; }

// ---------------------------------------------------------------------------
// shapes known on the host
// ---------------------------------------------------------------------------
struct Shape {
  int T, ndoc, max_seqlen, hq, hkv, G, d, dp, K;
  int window, dilation;  // block pattern: blocks j - dilation * u, u = 1..window, always kept
  int nb_bound;  // upper bound of KV blocks in the batch: ceil(T/128) + ndoc
  int nchunks;   // regroup chunks
  float softmax_scale, proxy_scale, kl_weight;
  int qc_blocks; // KV blocks per query chunk (qchunk_of)
  int nqchunks;  // query chunks of the slot partials
  int qc_tokens; // tokens of the largest query chunk: rows of the partial buffers
  bool test_stall_select;  // MSA_FLAG_TEST_STALL_SELECT
};

// ---------------------------------------------------------------------------
// Query chunks.  The per-slot partials of the forward (O, lse) and backward
// (dQ) take T * Hq * k * d * 2 and 4 bytes; to bound the workspace, one call
// processes the queries in chunks of whole KV blocks: chunk c holds the
// queries of global blocks [c * qcb, (c + 1) * qcb), so at most qcb * 128
// tokens (qcb = kQChunkBlocks unless the environment variable
// MSA_QUERY_CHUNK_BLOCKS sets a smaller positive value, used to test the
// chunked path on small batches).  Partial rows are indexed by token - t0.
// ---------------------------------------------------------------------------
constexpr int kQChunkBlocks = 2048;
struct QChunk {
  int b0, b1;  // global block range
  int t0, t1;  // token range
};
__device__ __forceinline__ int block_token_start(const int32_t* cu, const int32_t* cu_blocks,
                                                 int ndoc, int gb) {
  const int d = doc_of_block(cu_blocks, ndoc, gb);
  return __ldg(cu + d) + (gb - cu_blocks[d]) * kBlock;
}
// c < 0: the whole batch in one chunk.
__device__ __forceinline__ QChunk qchunk_of(const int32_t* cu, const int32_t* cu_blocks,
                                            int ndoc, int T, int nbt, int c, int qcb) {
  QChunk q;
  if (c < 0) {
    q.b0 = 0;
    q.b1 = nbt;
    q.t0 = 0;
    q.t1 = T;
    return q;
  }
  q.b0 = min(nbt, c * qcb);
  q.b1 = min(nbt, q.b0 + qcb);
  q.t0 = q.b0 < nbt ? block_token_start(cu, cu_blocks, ndoc, q.b0) : T;
  q.t1 = q.b1 < nbt ? block_token_start(cu, cu_blocks, ndoc, q.b1) : T;
  return q;
}
// First index i in [lo, hi) of a token-ascending list (ent = token << 4 | slot)
// with token >= t, or hi.
__device__ __forceinline__ int lower_bound_token(const uint32_t* ent, int lo, int hi, int t) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((int)(__ldg(ent + mid) >> 4) < t) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Workspace carve-up (byte offsets, 256-byte aligned).
struct Workspace {
  size_t cu_blocks, chunk_range, cnt, row_ptr, ent;          // metadata + regroup CSR
  size_t o_part, o_meta;                  // forward slot partials: int16 rows, {lse, scale}
  size_t dsum, dq_part, kl_part, rec;     // backward (dQ partials fp32)
  size_t total;
};
enum WsKind { kWsSelect = 0, kWsFwd = 1, kWsBwd = 2 };
Workspace workspace_layout(const Shape& s, WsKind kind);

// Host-side parameter checks shared by the entry points (fills `s` on MSA_OK).
msa_status check_params(const msa_params* p, Shape* s);
// Address of the current device's status word.
cudaError_t status_ptr(unsigned** out);
// Adds to the process-wide count of launched kernels (msa_launch_count).
void add_launches(uint64_t n);

// ---------------------------------------------------------------------------
// launchers (return cudaGetLastError() of their launches)
// ---------------------------------------------------------------------------
struct TmapEncoder;  // opaque; resolves cuTensorMapEncodeTiled once
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid,
                         uint64_t outer, uint32_t box_inner, uint32_t box_mid, uint32_t box_outer,
                         int swizzle_bytes);

cudaError_t launch_meta(const Shape& s, const int32_t* cu_seqlens, int32_t* cu_blocks,
                        unsigned* status, cudaStream_t st);
// with_arg: the selector also finds the argmax of every kept block; without
// it only the diagonal block's, and launch_sel_arg fills in the others.
cudaError_t launch_select(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                          const uint16_t* q_p, const uint16_t* k_p, int32_t* sel_idx,
                          float* sel_score, uint8_t* sel_arg, float* plse, uint8_t* tie,
                          bool with_arg, unsigned* status, cudaStream_t st);
cudaError_t launch_sel_arg(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                           const int32_t* row_ptr, const uint32_t* ent, const uint16_t* q_p,
                           const uint16_t* k_p, uint8_t* sel_arg, unsigned* status,
                           cudaStream_t st);
cudaError_t launch_regroup(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                           const int32_t* sel_idx, int32_t* chunk_range, uint32_t* cnt,
                           int32_t* row_ptr, uint32_t* ent, unsigned* status, cudaStream_t st);
cudaError_t launch_fwd(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                       const int32_t* row_ptr, const uint32_t* ent, const uint16_t* q,
                       const uint16_t* k, const uint16_t* v, int16_t* o_part, float2* o_meta,
                       int chunk, unsigned* status, cudaStream_t st);
cudaError_t launch_fwd_merge(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                             const int16_t* o_part, const float2* o_meta, uint16_t* o,
                             uint16_t* o_res, float* lse, float* mass, int chunk,
                             cudaStream_t st);  // chunk as launch_bwd_reduce
cudaError_t launch_bwd_pre(const Shape& s, const uint16_t* o, const uint16_t* o_res,
                           const uint16_t* dO, float* dsum, cudaStream_t st);
cudaError_t launch_bwd(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                       const int32_t* row_ptr, const uint32_t* ent, uint8_t* rec,
                       const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const uint16_t* q_p, const uint16_t* dO, const float* lse,
                       const float* dsum, const float* mass, const float* sel_score,
                       const uint8_t* sel_arg, const float* plse, float* dq_part, float* dk,
                       float* dv, float* dk_p, int chunk, unsigned* status, cudaStream_t st);
// chunk < 0: one call over all tokens; otherwise the queries of chunk `chunk`
// (partials indexed by token - t0); the KL scalar is produced when `last`.
cudaError_t launch_bwd_reduce(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                              const float* dq_part, const int32_t* sel_idx,
                              const float* sel_score, const uint8_t* sel_arg, const float* plse,
                              const float* mass, const uint16_t* k_p, float* dq, float* dq_p,
                              double* kl_part, double* kl_loss, int chunk, bool last,
                              cudaStream_t st);
int bwd_reduce_blocks(const Shape& s);

}  // namespace msa

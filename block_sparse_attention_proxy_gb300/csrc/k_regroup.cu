// Varlen metadata and the MoBA-style regroup.
//
// Regroup ("MoBA varlen trick", Flash-MSA summary on socker-news.uzaya.net,
// 要約): for every (KV group g, KV block) the list of (token, slot) pairs whose
// selection picked that block off the diagonal, as a CSR.  Lists are in
// ascending token order, so the result is deterministic: a chunked stable
// counting sort (count per chunk -> prefix over chunks -> sequential scatter).
#include "msa_internal.cuh"

namespace msa {
namespace {

// cu_blocks[d] = number of 128-token blocks in documents 0..d-1, plus checks of
// cu_seqlens (first 0, last T, lengths in [0, max_seqlen]).  One CTA.
__global__ void __launch_bounds__(1024) k_meta(const int32_t* __restrict__ cu, int ndoc, int T,
                                               int max_seqlen, int nb_bound,
                                               int32_t* __restrict__ cu_blocks,
                                               unsigned* status) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  __shared__ int bad_s;
  if (tid == 0) {
    carry_s = 0;
    bad_s = 0;
    cu_blocks[0] = 0;
    if (cu[0] != 0 || cu[ndoc] != T) bad_s = 1;
  }
  __syncthreads();
  for (int base = 0; base < ndoc; base += 1024) {
    const int d = base + tid;
    int nb = 0;
    if (d < ndoc) {
      int L = cu[d + 1] - cu[d];
      if (L < 0 || L > max_seqlen) {
        bad_s = 1;
        L = L < 0 ? 0 : max_seqlen;
      }
      nb = (L + kBlock - 1) / kBlock;
    }
    int x = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
      int y = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int z = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += z;
      }
      warp_tot[lane] = y;
    }
    __syncthreads();
    const int incl = x + (w > 0 ? warp_tot[w - 1] : 0);
    const int carry = carry_s;
    if (d < ndoc) cu_blocks[d + 1] = min(carry + incl, nb_bound);
    __syncthreads();
    if (tid == 1023) carry_s = carry + incl;
    __syncthreads();
  }
  // cu_blocks[ndoc + 1] = 1 when cu_seqlens is well formed; every later kernel
  // of the call reads it and does nothing otherwise.
  if (tid == 0) {
    cu_blocks[ndoc + 1] = bad_s ? 0 : 1;
    if (bad_s) set_status(status, MSA_ERR_DEVICE_CHECK);
  }
}

// Checks the structure of one selection row (K slots): slots below
// sd = min(j, K-1) hold strictly ascending blocks in [0, j), slot sd holds the
// diagonal j, the rest hold -1.  Rows failing the check are skipped by both
// regroup passes (identically), and flagged.
__device__ __forceinline__ bool row_ok_serial(const int32_t* row, int K, int j) {
  const int sd = min(j, K - 1);
  int prev = -1;
  for (int s = 0; s < K; ++s) {
    const int b = row[s];
    if (s < sd) {
      if (b <= prev || b >= j) return false;
      prev = b;
    } else if (s == sd) {
      if (b != j) return false;
    } else if (b != -1) {
      return false;
    }
  }
  return true;
}

// Range [lo, hi) of global blocks the tokens of chunk c can select.
__device__ __forceinline__ void chunk_block_range(const int32_t* cu, const int32_t* cu_blocks,
                                                  int ndoc, int t0, int t1, int nb_bound,
                                                  int& lo, int& hi) {
  const int d0 = doc_of_token(cu, ndoc, t0), d1 = doc_of_token(cu, ndoc, t1 - 1);
  lo = min(cu_blocks[d0], nb_bound);
  hi = min(cu_blocks[d1] + (t1 - 1 - cu[d1]) / kBlock + 1, nb_bound);
  if (hi < lo) hi = lo;
}

__global__ void __launch_bounds__(256) k_rg_count(const int32_t* __restrict__ cu,
                                                  const int32_t* __restrict__ cu_blocks, int ndoc,
                                                  int T, int Hkv, int K, int nbs,
                                                  const int32_t* __restrict__ sel_idx,
                                                  int32_t* __restrict__ chunk_range,
                                                  uint32_t* __restrict__ cnt, unsigned* status) {
  extern __shared__ uint32_t cnt_s[];
  if (!cu_blocks[ndoc + 1]) return;
  const int c = blockIdx.x, g = blockIdx.y;
  const int t0 = c * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  int lo, hi;
  chunk_block_range(cu, cu_blocks, ndoc, t0, t1, nbs, lo, hi);
  const int R = hi - lo;
  for (int i = threadIdx.x; i < R; i += blockDim.x) cnt_s[i] = 0;
  __syncthreads();
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    const int d = doc_of_token(cu, ndoc, t);
    const int j = (t - cu[d]) / kBlock;
    const int32_t* row = sel_idx + ((size_t)t * Hkv + g) * K;
    if (!row_ok_serial(row, K, j)) {
      set_status(status, MSA_ERR_DEVICE_CHECK);
      continue;
    }
    const int sd = min(j, K - 1);
    const int gbd = cu_blocks[d];
    for (int s = 0; s < sd; ++s) {
      const int gbi = gbd + row[s] - lo;
      if (gbi >= 0 && gbi < R) atomicAdd(&cnt_s[gbi], 1u);
    }
  }
  __syncthreads();
  uint32_t* out = cnt + ((size_t)c * Hkv + g) * nbs + lo;
  for (int i = threadIdx.x; i < R; i += blockDim.x) out[i] = cnt_s[i];
  if (g == 0 && threadIdx.x == 0) {
    chunk_range[2 * c] = lo;
    chunk_range[2 * c + 1] = hi;
  }
}

// Per (g, block): exclusive prefix of the chunk counts (in place) and the
// block's total, written to row_ptr[1 + g*nbs + gb].
__global__ void __launch_bounds__(256) k_rg_scan(int nchunks, int Hkv, int nbs,
                                                 const int32_t* __restrict__ chunk_range,
                                                 uint32_t* __restrict__ cnt,
                                                 int32_t* __restrict__ row_ptr) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= Hkv * nbs) return;
  const int g = idx / nbs, gb = idx - g * nbs;
  uint32_t run = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int lo = chunk_range[2 * c], hi = chunk_range[2 * c + 1];
    if (gb >= lo && gb < hi) {
      uint32_t* p = cnt + ((size_t)c * Hkv + g) * nbs + gb;
      const uint32_t v = *p;
      *p = run;
      run += v;
    }
  }
  row_ptr[1 + idx] = (int32_t)run;
}

// In-place inclusive scan of row_ptr[1..n] (one CTA), row_ptr[0] = 0.
__global__ void __launch_bounds__(1024) k_rg_rowptr(int n, int32_t* __restrict__ row_ptr) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + 1023) / 1024;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int s = 0;
  for (int i = b0; i < b1; ++i) s += row_ptr[1 + i];
  int x = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int y = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    warp_tot[lane] = y;
  }
  __syncthreads();
  int run = x - s + (w > 0 ? warp_tot[w - 1] : 0);  // exclusive prefix of this segment
  for (int i = b0; i < b1; ++i) {
    run += row_ptr[1 + i];
    row_ptr[1 + i] = run;
  }
  if (tid == 0) row_ptr[0] = 0;
}

// One warp per (chunk, g): walks the chunk's tokens in order, lane s handling
// slot s; the slots of one token name distinct blocks, so no two lanes bump the
// same counter in a step.
__global__ void __launch_bounds__(32) k_rg_scatter(const int32_t* __restrict__ cu,
                                                   const int32_t* __restrict__ cu_blocks, int ndoc,
                                                   int T, int Hkv, int K, int nbs,
                                                   const int32_t* __restrict__ sel_idx,
                                                   const int32_t* __restrict__ chunk_range,
                                                   const uint32_t* __restrict__ cnt,
                                                   const int32_t* __restrict__ row_ptr,
                                                   uint32_t* __restrict__ ent) {
  extern __shared__ uint32_t off_s[];
  if (!cu_blocks[ndoc + 1]) return;
  const int c = blockIdx.x, g = blockIdx.y, lane = threadIdx.x;
  const int t0 = c * kChunkTokens, t1 = min(T, t0 + kChunkTokens);
  const int lo = chunk_range[2 * c], hi = chunk_range[2 * c + 1];
  const int R = hi - lo;
  const uint32_t* cc = cnt + ((size_t)c * Hkv + g) * nbs + lo;
  const int32_t* rp = row_ptr + (size_t)g * nbs + lo;
  for (int i = lane; i < R; i += 32) off_s[i] = (uint32_t)rp[i] + cc[i];
  __syncwarp();
  int d = doc_of_token(cu, ndoc, t0);
  int dstart = cu[d], dend = cu[d + 1], gbd = cu_blocks[d];
  // The selection rows of kAhead tokens are loaded together (independent
  // loads in flight), then the tokens are scattered one by one in order.
  constexpr int kAhead = 16;
  for (int tb = t0; tb < t1; tb += kAhead) {
    int bq[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int t = tb + u;
      bq[u] = (t < t1 && lane < K) ? __ldg(sel_idx + ((size_t)t * Hkv + g) * K + lane) : -1;
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int t = tb + u;
      if (t >= t1) break;  // warp-uniform
      while (t >= dend && d + 1 < ndoc) {
        ++d;
        dstart = dend;
        dend = cu[d + 1];
        gbd = cu_blocks[d];
      }
      const int j = (t - dstart) / kBlock;
      const int sd = min(j, K - 1);
      const int b = bq[u];
      // identical structural check to row_ok_serial, done across lanes
      const int prev = __shfl_up_sync(0xffffffffu, b, 1);
      bool ok = true;
      if (lane < K) {
        if (lane < sd) ok = b >= 0 && b < j && (lane == 0 || b > prev);
        else if (lane == sd) ok = b == j;
        else ok = b == -1;
      }
      if (__all_sync(0xffffffffu, ok) && lane < sd) {
        const int gbi = gbd + b - lo;
        if (gbi >= 0 && gbi < R) {
          const uint32_t pos = off_s[gbi];
          off_s[gbi] = pos + 1;
          ent[pos] = ((uint32_t)t << 4) | (uint32_t)lane;
        }
      }
      __syncwarp();
    }
  }
}

}  // namespace

cudaError_t launch_meta(const Shape& s, const int32_t* cu_seqlens, int32_t* cu_blocks,
                        unsigned* status, cudaStream_t st) {
  k_meta<<<1, 1024, 0, st>>>(cu_seqlens, s.ndoc, s.T, s.max_seqlen, s.nb_bound, cu_blocks,
                             status);
  return cudaGetLastError();
}

cudaError_t launch_regroup(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                           const int32_t* sel_idx, int32_t* chunk_range, uint32_t* cnt,
                           int32_t* row_ptr, uint32_t* ent, unsigned* status, cudaStream_t st) {
  const int nbs = s.nb_bound;
  const size_t smem = (size_t)nbs * sizeof(uint32_t);
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_rg_count, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_rg_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  dim3 grid(s.nchunks, s.hkv);
  k_rg_count<<<grid, 256, smem, st>>>(cu_seqlens, cu_blocks, s.ndoc, s.T, s.hkv, s.K, nbs,
                                      sel_idx, chunk_range, cnt, status);
  const int n = s.hkv * nbs;
  k_rg_scan<<<(n + 255) / 256, 256, 0, st>>>(s.nchunks, s.hkv, nbs, chunk_range, cnt, row_ptr);
  k_rg_rowptr<<<1, 1024, 0, st>>>(n, row_ptr);
  k_rg_scatter<<<grid, 32, smem, st>>>(cu_seqlens, cu_blocks, s.ndoc, s.T, s.hkv, s.K, nbs,
                                       sel_idx, chunk_range, cnt, row_ptr, ent);
  return cudaGetLastError();
}

}  // namespace msa

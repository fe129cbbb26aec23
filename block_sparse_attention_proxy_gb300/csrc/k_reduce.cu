// Memory-bound epilogues of the forward and backward passes.
//
//   k_fwd_merge   per (token, group): log-sum-exp merge of the per-slot partials
//                 of every head (O as 16-bit fixed point with a per-row scale,
//                 lse), and the target mass of the proxy loss
//                 m_b = (1/G) sum_h exp(lse_{h,b} - LSE_h) per selected block.
//                 It also writes o_res = bf16(O - bf16(O)), the rounding residual
//                 of the bf16 output, so the backward can form D from ~16 bits of O.
//   k_bwd_pre     D = rowsum(dO * (o + o_res)) per (token, head).
//   k_bwd_reduce  per (token, group): dQ = sum over slots of the fp32 dQ partials
//                 (fixed order); the proxy gradient
//                 dq_p = proxy_scale * sum_b kl_weight (p_b - m_b) k_p[a_b];
//                 the KL term sum_b m_b (log m_b - log p_b), reduced per CTA in a
//                 fixed order, then over CTAs by k_kl_final (fp64).
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kRedWarps = 8;

__device__ __forceinline__ int nsel_of(const int32_t* cu, int ndoc, int t, int K) {
  const int d = doc_of_token(cu, ndoc, t);
  const int j = (t - __ldg(cu + d)) / kBlock;
  return min(j, K - 1) + 1;
}

template <int D>
__global__ void __launch_bounds__(kRedWarps * 32)
    k_fwd_merge(int T, int ndoc, const int32_t* __restrict__ cu,
                const int32_t* __restrict__ cu_blocks, int nb_bound, int chunk, int qcb, int hkv,
                int G, int K, const int16_t* __restrict__ o_part,
                const float2* __restrict__ o_meta, uint16_t* __restrict__ o,
                uint16_t* __restrict__ o_res, float* __restrict__ lse, float* __restrict__ mass) {
  constexpr int PER = D / 32;  // head-dim elements per lane
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kRedWarps + (threadIdx.x >> 5);
  if (wid >= (long long)T * hkv) return;
  const int t = (int)(wid / hkv), g = (int)(wid % hkv);
  // partial rows of this launch's query chunk are indexed by token - t0
  int t0 = 0;
  if (chunk >= 0) {
    const QChunk qc =
        qchunk_of(cu, cu_blocks, ndoc, T, min(cu_blocks[ndoc], nb_bound), chunk, qcb);
    if (t < qc.t0 || t >= qc.t1) return;
    t0 = qc.t0;
  }
  const int hq = hkv * G;
  const int nsel = nsel_of(cu, ndoc, t, K);
  float macc = 0.f;
  for (int hh = 0; hh < G; ++hh) {
    const size_t row = (size_t)t * hq + g * G + hh;
    const size_t prow = (size_t)(t - t0) * hq + g * G + hh;
    const float2 meta = lane < nsel ? __ldg(o_meta + prow * K + lane)
                                    : make_float2(-INFINITY, 0.f);
    // every slot's partial is requested before any is used
    const int16_t* src = o_part + prow * K * (size_t)D + lane * PER;
    uint32_t x[kMaxTopK][PER / 2];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      if (s < nsel) {
        if (PER == 4) {
          const uint2 v2 = __ldg(reinterpret_cast<const uint2*>(src + (size_t)s * D));
          x[s][0] = v2.x;
          x[s][PER / 2 - 1] = v2.y;
        } else {
          x[s][0] = __ldg(reinterpret_cast<const unsigned int*>(src + (size_t)s * D));
        }
      }
    }
    const float ls = meta.x;
    const float mx = warp_max(ls);
    const float se = warp_sum(lane < nsel ? __expf(ls - mx) : 0.f);
    const float LSE = mx + __logf(se);
    const float w = lane < nsel ? __expf(ls - LSE) : 0.f;
    macc += w;
    const float wq = w * meta.y;  // merge weight times the slot row's scale
    float acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      const float ws = __shfl_sync(0xffffffffu, wq, s);
      if (s < nsel) {
#pragma unroll
        for (int u = 0; u < PER / 2; ++u) {
          acc[2 * u] = fmaf(ws, q16_lo(x[s][u]), acc[2 * u]);
          acc[2 * u + 1] = fmaf(ws, q16_hi(x[s][u]), acc[2 * u + 1]);
        }
      }
    }
    uint16_t* dst = o + row * D + lane * PER;
    uint16_t* rdst = o_res + row * D + lane * PER;
    uint32_t hi[PER / 2], lo[PER / 2];
#pragma unroll
    for (int u = 0; u < PER / 2; ++u) {
      hi[u] = pack_bf16(acc[2 * u], acc[2 * u + 1]);
      lo[u] = pack_bf16(acc[2 * u] - bf16_lo(hi[u]), acc[2 * u + 1] - bf16_hi(hi[u]));
    }
    if (PER == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(hi[0], hi[PER / 2 - 1]);
      *reinterpret_cast<uint2*>(rdst) = make_uint2(lo[0], lo[PER / 2 - 1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst) = hi[0];
      *reinterpret_cast<uint32_t*>(rdst) = lo[0];
    }
    if (lane == 0) lse[row] = LSE;
  }
  if (lane < K) mass[((size_t)t * hkv + g) * K + lane] = lane < nsel ? macc / (float)G : 0.f;
}

template <int D>
__global__ void __launch_bounds__(256) k_bwd_pre(long long rows, const uint16_t* __restrict__ o,
                                                 const uint16_t* __restrict__ o_res,
                                                 const uint16_t* __restrict__ dO,
                                                 float* __restrict__ dsum) {
  // D/8 lanes per (token, head) row, 16 bytes of o, o_res and dO per lane; a warp
  // takes kPreIters row groups and requests all of them before summing
  constexpr int LPR = D / 8, RPW = 32 / LPR, kPreIters = 4;
  const int lane = threadIdx.x & 31;
  const long long r0 =
      ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * (RPW * kPreIters) + lane / LPR;
  const int c = (lane % LPR) * 8;
  uint4 x[kPreIters], e[kPreIters], y[kPreIters];
#pragma unroll
  for (int u = 0; u < kPreIters; ++u) {
    const long long r = r0 + (long long)u * RPW;
    x[u] = e[u] = y[u] = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
      x[u] = __ldg(reinterpret_cast<const uint4*>(o + r * D + c));
      e[u] = __ldg(reinterpret_cast<const uint4*>(o_res + r * D + c));
      y[u] = __ldg(reinterpret_cast<const uint4*>(dO + r * D + c));
    }
  }
#pragma unroll
  for (int u = 0; u < kPreIters; ++u) {
    const long long r = r0 + (long long)u * RPW;
    const uint32_t xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
    const uint32_t es[4] = {e[u].x, e[u].y, e[u].z, e[u].w};
    const uint32_t ys[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      s += (bf16_lo(xs[q]) + bf16_lo(es[q])) * bf16_lo(ys[q]) +
           (bf16_hi(xs[q]) + bf16_hi(es[q])) * bf16_hi(ys[q]);
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (r < rows && lane % LPR == 0) dsum[r] = s;
  }
}

template <int D, int DP>
__global__ void __launch_bounds__(kRedWarps * 32)
    k_bwd_reduce(int T, int ndoc, const int32_t* __restrict__ cu,
                 const int32_t* __restrict__ cu_blocks, int nb_bound, int chunk, int qcb, int hkv,
                 int G, int K, float proxy_scale, float kl_weight, const float* __restrict__ dq_part,
                 const int32_t* __restrict__ sel_idx, const float* __restrict__ sel_score,
                 const uint8_t* __restrict__ sel_arg, const float* __restrict__ plse,
                 const float* __restrict__ mass, const uint16_t* __restrict__ k_p,
                 float* __restrict__ dq, float* __restrict__ dq_p, double* __restrict__ kl_part) {
  constexpr int PER = D / 32;
  constexpr int PPER = DP / 32;
  __shared__ double wkl[kRedWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const long long wid = (long long)blockIdx.x * kRedWarps + w;
  double kl_w = 0.0;
  // partial rows of this launch's query chunk are indexed by token - t0
  int t0 = 0, t1 = T;
  if (chunk >= 0) {
    const QChunk qc =
        qchunk_of(cu, cu_blocks, ndoc, T, min(cu_blocks[ndoc], nb_bound), chunk, qcb);
    t0 = qc.t0;
    t1 = qc.t1;
  }
  const int tw = (int)(wid / hkv);
  if (wid < (long long)T * hkv && tw >= t0 && tw < t1) {
    const int t = tw, g = (int)(wid % hkv);
    const int hq = hkv * G;
    const int d = doc_of_token(cu, ndoc, t);
    const int dstart = __ldg(cu + d);
    const int j = (t - dstart) / kBlock;
    const int nsel = min(j, K - 1) + 1;
    // ---- dQ: fixed-order sum of the slot partials ----
    for (int hh = 0; hh < G; ++hh) {
      const size_t row = (size_t)t * hq + g * G + hh;
      const float* src = dq_part + ((size_t)(t - t0) * hq + g * G + hh) * K * (size_t)D + lane * PER;
      float acc[PER];
#pragma unroll
      for (int u = 0; u < PER; ++u) acc[u] = 0.f;
      for (int s = 0; s < nsel; ++s) {
        if (PER == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(src + (size_t)s * D));
          acc[0] += x.x;
          acc[1] += x.y;
          acc[PER > 2 ? 2 : 0] += x.z;
          acc[PER > 3 ? 3 : 0] += x.w;
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(src + (size_t)s * D));
          acc[0] += x.x;
          acc[1] += x.y;
        }
      }
      float* dst = dq + row * D + lane * PER;
      if (PER == 4)
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[PER > 2 ? 2 : 0], acc[PER > 3 ? 3 : 0]);
      else
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
    }
    // ---- proxy: g_b, KL term, dq_p ----
    const size_t e0 = ((size_t)t * hkv + g) * K;
    const float pl = __ldg(plse + (size_t)t * hkv + g);
    float gs = 0.f;
    int key = 0;
    double term = 0.0;
    if (lane < nsel) {
      const float p = __expf(__ldg(sel_score + e0 + lane) - pl);
      const float m = __ldg(mass + e0 + lane);
      gs = kl_weight * (p - m);
      if (m > 0.f) term = (double)m * (log((double)m) - ((double)__ldg(sel_score + e0 + lane) - (double)pl));
      const int b = __ldg(sel_idx + e0 + lane);
      key = dstart + b * kBlock + __ldg(sel_arg + e0 + lane);
      if (b < 0 || b > j || key < 0 || key >= T) {  // malformed selection: contributes nothing
        gs = 0.f;
        key = t;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
    kl_w = term;
    float acc[PPER];
#pragma unroll
    for (int u = 0; u < PPER; ++u) acc[u] = 0.f;
    for (int s = 0; s < nsel; ++s) {
      const float gsv = __shfl_sync(0xffffffffu, gs, s);
      const int ky = __shfl_sync(0xffffffffu, key, s);
      const uint16_t* kr = k_p + ((size_t)ky * hkv + g) * DP + lane * PPER;
      if (PPER == 2) {
        const uint32_t x = __ldg(reinterpret_cast<const unsigned int*>(kr));
        acc[0] = fmaf(gsv, bf16_lo(x), acc[0]);
        acc[PPER - 1] = fmaf(gsv, bf16_hi(x), acc[PPER - 1]);
      } else {
        acc[0] = fmaf(gsv, __uint_as_float((uint32_t)__ldg(kr) << 16), acc[0]);
      }
    }
    float* dst = dq_p + ((size_t)t * hkv + g) * DP + lane * PPER;
#pragma unroll
    for (int u = 0; u < PPER; ++u) dst[u] = proxy_scale * acc[u];
  }
  if (lane == 0) wkl[w] = kl_w;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < kRedWarps; ++i) s += wkl[i];
    // a CTA may hold tokens of two query chunks: later chunks add (fixed order)
    kl_part[blockIdx.x] = chunk > 0 ? kl_part[blockIdx.x] + s : s;
  }
}

__global__ void __launch_bounds__(1024) k_kl_final(int n, const double* __restrict__ part,
                                                   float kl_weight, double* __restrict__ out) {
  // fixed-order tree: each thread sums a contiguous segment, then thread 0 sums the segments
  __shared__ double seg[1024];
  const int per = (n + 1023) / 1024;
  const int b0 = min(n, (int)threadIdx.x * per), b1 = min(n, b0 + per);
  double s = 0.0;
  for (int i = b0; i < b1; ++i) s += part[i];
  seg[threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int i = 0; i < 1024; ++i) tot += seg[i];
    *out = (double)kl_weight * tot;
  }
}

}  // namespace

cudaError_t launch_fwd_merge(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                             const int16_t* o_part, const float2* o_meta, uint16_t* o,
                             uint16_t* o_res, float* lse, float* mass, int chunk,
                             cudaStream_t st) {
  const long long warps = (long long)s.T * s.hkv;
  const int blocks = (int)((warps + kRedWarps - 1) / kRedWarps);
  if (s.d == 128)
    k_fwd_merge<128><<<blocks, kRedWarps * 32, 0, st>>>(s.T, s.ndoc, cu_seqlens, cu_blocks,
                                                         s.nb_bound, chunk, s.qc_blocks, s.hkv,
                                                         s.G, s.K, o_part, o_meta, o, o_res,
                                                         lse, mass);
  else
    k_fwd_merge<64><<<blocks, kRedWarps * 32, 0, st>>>(s.T, s.ndoc, cu_seqlens, cu_blocks,
                                                        s.nb_bound, chunk, s.qc_blocks, s.hkv,
                                                        s.G, s.K, o_part, o_meta, o, o_res,
                                                        lse, mass);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const Shape& s, const uint16_t* o, const uint16_t* o_res,
                           const uint16_t* dO, float* dsum, cudaStream_t st) {
  const long long rows = (long long)s.T * s.hq;
  const long long per_cta = 8LL * 4 * (32 / (s.d / 8));  // 8 warps x 4 row groups x rows per group
  const int blocks = (int)((rows + per_cta - 1) / per_cta);
  if (s.d == 128)
    k_bwd_pre<128><<<blocks, 256, 0, st>>>(rows, o, o_res, dO, dsum);
  else
    k_bwd_pre<64><<<blocks, 256, 0, st>>>(rows, o, o_res, dO, dsum);
  return cudaGetLastError();
}

int bwd_reduce_blocks(const Shape& s) {
  const long long warps = (long long)s.T * s.hkv;
  return (int)((warps + kRedWarps - 1) / kRedWarps);
}

cudaError_t launch_bwd_reduce(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                              const float* dq_part, const int32_t* sel_idx,
                              const float* sel_score, const uint8_t* sel_arg, const float* plse,
                              const float* mass, const uint16_t* k_p, float* dq, float* dq_p,
                              double* kl_part, double* kl_loss, int chunk, bool last,
                              cudaStream_t st) {
  const int blocks = bwd_reduce_blocks(s);
#define MSA_RED(DD, PP)                                                                         \
  k_bwd_reduce<DD, PP><<<blocks, kRedWarps * 32, 0, st>>>(                                      \
      s.T, s.ndoc, cu_seqlens, cu_blocks, s.nb_bound, chunk, s.qc_blocks, s.hkv, s.G, s.K,      \
      s.proxy_scale, s.kl_weight, dq_part, sel_idx, sel_score, sel_arg, plse, mass, k_p, dq,     \
      dq_p, kl_part)
  if (s.d == 128 && s.dp == 64) MSA_RED(128, 64);
  else if (s.d == 128) MSA_RED(128, 32);
  else if (s.dp == 64) MSA_RED(64, 64);
  else MSA_RED(64, 32);
#undef MSA_RED
  if (last) k_kl_final<<<1, 1024, 0, st>>>(blocks, kl_part, s.kl_weight, kl_loss);
  return cudaGetLastError();
}

}  // namespace msa

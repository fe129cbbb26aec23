// Block-sparse attention forward, KV-major.
//
// The Flash-MSA summary (socker-news.uzaya.net, 要約) runs sparse attention
// through FlashAttention with MoBA's varlen trick: the queries that chose a
// KV block are gathered and attend to that block as one varlen problem.  Here
// one CTA owns one (KV group g, KV block b): K_b and V_b are staged once by
// TMA, then tiles of 128 rows = 128/G tokens x G heads are processed:
//   * first the block's own queries (the diagonal slot, causal inside the block),
//   * then the gathered queries from the regroup CSR (full block, no mask).
// Per tile: S = Q K^T on tcgen05 into TMEM, exact softmax over the block's 128
// keys (one TMEM lane = one row), P to shared memory as two bf16 operands
// (hi = bf16(P), lo = bf16(P - hi), so O keeps ~16 mantissa bits of P; the
// backward's D = rowsum(dO * O) needs that), O = P_hi V + P_lo V into TMEM,
// and the normalised partial O_slot and lse_slot (both fp32) are written per
// (token, head, slot).  The merge kernel combines the slots by log-sum-exp.
//
// Roles (192 threads): warps 0-3 softmax/epilogue, warp 4 TMA producer,
// warp 5 MMA issuer.  Two Q buffers, two S and two O accumulators, one P buffer
// (the epilogue rewrites P only after the previous P V has completed).
#include <cfloat>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kFwdThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

struct FwdArgs {
  const int32_t* cu;
  const int32_t* cu_blocks;
  const int32_t* row_ptr;
  const uint32_t* ent;
  int ndoc, T, hq, hkv, K, nb_bound;
  float scale;
  float* o_part;
  float* lse_part;
  unsigned* status;
};

template <int D, int G>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  constexpr int TPT = 128 / G;         // tokens per tile
  constexpr int NCH = D / 64;          // 64-column chunks of a head row
  constexpr int kTile = 128 * D * 2;   // bytes of a 128-row, D-column bf16 tile
  constexpr int kPTile = 128 * 128 * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTile;
  uint8_t* sQ = sV + kTile;       // [2]
  uint8_t* sP = sQ + 2 * kTile;   // hi part of P
  uint8_t* sPl = sP + kPTile;     // lo part of P
  uint64_t* bars = reinterpret_cast<uint64_t*>(sPl + kPTile);
  // 0 kv_full | 1,2 q_full | 3,4 q_empty | 5,6 s_full | 7,8 s_empty | 9 p_full (10 unused) |
  // 11,12 o_full | 13,14 o_empty
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item ----
  if (!a.cu_blocks[a.ndoc + 1]) return;  // malformed cu_seqlens (flagged by k_meta)
  const int nbt = min(a.cu_blocks[a.ndoc], a.nb_bound);
  const int g = blockIdx.x % a.hkv;
  const int gb = (int)(blockIdx.x / a.hkv);
  if (gb >= nbt) return;
  const int d = doc_of_block(a.cu_blocks, a.ndoc, gb);
  const int j = gb - a.cu_blocks[d];
  const int dstart = a.cu[d];
  const int L = a.cu[d + 1] - dstart;
  const int kstart = dstart + j * kBlock;
  const int nkeys = min(kBlock, L - j * kBlock);
  const int lbeg = a.row_ptr[g * a.nb_bound + gb];
  const int lcnt = a.row_ptr[g * a.nb_bound + gb + 1] - lbeg;
  const int ndiag = (nkeys + TPT - 1) / TPT;
  const int ntiles = ndiag + (lcnt + TPT - 1) / TPT;
  const int slot_diag = min(j, a.K - 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 15; ++i) {
      const bool four = (i == 7 || i == 8 || i == 9 || i == 10 || i == 13 || i == 14);
      mbar_init(bar(i), four ? 4 : 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(tslot);

  // token of tile row-group i of tile n (T = out of range -> TMA zero fill)
  auto tile_token = [&](int n, int i, int& t, int& slot) -> bool {
    if (n < ndiag) {
      const int qi = n * TPT + i;
      t = kstart + qi;
      slot = slot_diag;
      return qi < nkeys && t < a.T;
    }
    const int m = (n - ndiag) * TPT + i;
    if (m >= lcnt) {
      t = a.T;
      slot = 0;
      return false;
    }
    const uint32_t e = __ldg(a.ent + lbeg + m);
    t = (int)(e >> 4);
    slot = (int)(e & 15u);
    return t < a.T;
  };

  if (warp == 4) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(0), 2 * kTile);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d(smem_u32(sK + c * 16384), &tm_k, bar(0), 64 * c, g, kstart);
        tma_load_3d(smem_u32(sV + c * 16384), &tm_v, bar(0), 64 * c, g, kstart);
      }
    }
    for (int n = 0; n < ntiles; ++n) {
      const int buf = n & 1;
      if (n >= 2 && !wait_bar_warp(bar(3 + buf), ((n >> 1) & 1) ^ 1, abort_flag, a.status,
                                   wait_site(kKerFwd, 3 + buf, n)))
        break;
      if (lane == 0) mbar_arrive_expect_tx(bar(1 + buf), kTile);
      __syncwarp();
      const uint32_t qb = smem_u32(sQ + buf * kTile);
      for (int i = lane; i < TPT; i += 32) {
        int t, slot;
        if (!tile_token(n, i, t, slot)) t = a.T;
#pragma unroll
        for (int c = 0; c < NCH; ++c)
          tma_load_3d(qb + c * 16384 + i * G * 128, &tm_q, bar(1 + buf), 64 * c, g * G, t);
      }
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer ---------------------------------
    if (lane == 0) {
      constexpr uint32_t idS = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idO = make_idesc_bf16(128, D, false, true);
      bool ok = wait_bar(bar(0), 0, abort_flag, a.status, wait_site(kKerFwd, 0, 0));
      auto issue_s = [&](int n) -> bool {
        const int buf = n & 1, ph = (n >> 1) & 1;
        if (!wait_bar(bar(1 + buf), ph, abort_flag, a.status, wait_site(kKerFwd, 1 + buf, n)))
          return false;
        if (n >= 2 &&
            !wait_bar(bar(7 + buf), ph ^ 1, abort_flag, a.status, wait_site(kKerFwd, 7 + buf, n)))
          return false;
        tc_fence_after();
        const uint32_t q0 = smem_u32(sQ + buf * kTile), k0 = smem_u32(sK);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16(tbase + buf * 128, make_sdesc(q0 + off, 16, 1024, kLayoutSW128),
                    make_sdesc(k0 + off, 16, 1024, kLayoutSW128), idS, kk > 0);
        }
        umma_commit(bar(5 + buf));
        umma_commit(bar(3 + buf));
        return true;
      };
      if (ok && ntiles > 0) ok = issue_s(0);
      for (int n = 0; ok && n < ntiles; ++n) {
        const int buf = n & 1, ph = (n >> 1) & 1;
        if (n + 1 < ntiles && !issue_s(n + 1)) break;
        if (!wait_bar(bar(9), n & 1, abort_flag, a.status, wait_site(kKerFwd, 9, n))) break;
        if (n >= 2 &&
            !wait_bar(bar(13 + buf), ph ^ 1, abort_flag, a.status, wait_site(kKerFwd, 13 + buf, n)))
          break;
        tc_fence_after();
        const uint32_t p0 = smem_u32(sP), pl0 = smem_u32(sPl), v0 = smem_u32(sV);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t bd = make_sdesc(v0 + kk * 2048, 16384, 1024, kLayoutSW128);
          umma_bf16(tbase + 256 + buf * D, make_sdesc(p0 + off, 16, 1024, kLayoutSW128), bd, idO,
                    kk > 0);
          umma_bf16(tbase + 256 + buf * D, make_sdesc(pl0 + off, 16, 1024, kLayoutSW128), bd, idO,
                    1u);
        }
        umma_commit(bar(11 + buf));
      }
    }
  } else {
    // ------------------------------ softmax / epilogue --------------------------
    const int row = warp * 32 + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int ti = row / G, hl = row % G;
    const float sl2 = a.scale * kLog2e;
    for (int n = 0; n < ntiles; ++n) {
      const int buf = n & 1, ph = (n >> 1) & 1;
      int t, slot;
      const bool valid = tile_token(n, ti, t, slot);
      const bool diag = n < ndiag;
      const int qpos = n * TPT + ti;  // position inside the block (diagonal tiles)
      if (!wait_bar_warp(bar(5 + buf), ph, abort_flag, a.status, wait_site(kKerFwd, 5 + buf, n)))
        break;
      tc_fence_after();
      const uint32_t ts = tbase + lane_off + buf * 128;
      float mx = -FLT_MAX;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32f(ts + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const bool keep = !diag || (c * 32 + i <= qpos);
          mx = keep ? fmaxf(mx, v[i]) : mx;
        }
      }
      const float mb = mx * sl2;
      float l = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32f(ts + c * 32, v);
        uint32_t pk[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int k0 = c * 32 + 2 * i;
          const float p0 = (!diag || k0 <= qpos) ? exp2f(fmaf(v[2 * i], sl2, -mb)) : 0.f;
          const float p1 = (!diag || k0 + 1 <= qpos) ? exp2f(fmaf(v[2 * i + 1], sl2, -mb)) : 0.f;
          l += p0 + p1;
          pk[i] = pack_bf16(p0, p1);
          pl[i] = pack_bf16(p0 - bf16_lo(pk[i]), p1 - bf16_hi(pk[i]));
        }
        // 32 keys = 64 bytes = four 16-byte chunks of the row in key-chunk c/2
        const uint32_t cbase = (c >> 1) * 16384;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = cbase + sw128_offset((uint32_t)row, (uint32_t)((c & 1) * 4 + q));
          *reinterpret_cast<uint4*>(sP + off) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          *reinterpret_cast<uint4*>(sPl + off) =
              make_uint4(pl[4 * q], pl[4 * q + 1], pl[4 * q + 2], pl[4 * q + 3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(7 + buf));
        mbar_arrive(bar(9));
      }
      if (!wait_bar_warp(bar(11 + buf), ph, abort_flag, a.status, wait_site(kKerFwd, 11 + buf, n)))
        break;
      tc_fence_after();
      const float inv_l = 1.f / l;
      const uint32_t to = tbase + lane_off + 256 + buf * D;
      float* orow = a.o_part + (((size_t)t * a.hq + g * G + hl) * a.K + slot) * (size_t)D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32f(to + c * 32, v);
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(orow + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(v[4 * q] * inv_l, v[4 * q + 1] * inv_l, v[4 * q + 2] * inv_l,
                                 v[4 * q + 3] * inv_l);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(13 + buf));
      if (valid)
        a.lse_part[((size_t)t * a.hq + g * G + hl) * a.K + slot] = mx * a.scale + __logf(l);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, int G>
cudaError_t launch_fwd_t(const Shape& s, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const FwdArgs& a, cudaStream_t st) {
  const size_t smem = 1024 + 4 * (128 * D * 2) + 2 * (128 * 128 * 2) + 15 * 8 + 16;
  cudaError_t e = cudaFuncSetAttribute(k_fwd<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  k_fwd<D, G><<<s.nb_bound * s.hkv, kFwdThreads, smem, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const Shape& s, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const FwdArgs& a, cudaStream_t st) {
  switch (s.G) {
    case 1: return launch_fwd_t<D, 1>(s, mq, mk, mv, a, st);
    case 2: return launch_fwd_t<D, 2>(s, mq, mk, mv, a, st);
    case 4: return launch_fwd_t<D, 4>(s, mq, mk, mv, a, st);
    default: return launch_fwd_t<D, 8>(s, mq, mk, mv, a, st);
  }
}

}  // namespace

cudaError_t launch_fwd(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                       const int32_t* row_ptr, const uint32_t* ent, const uint16_t* q,
                       const uint16_t* k, const uint16_t* v, float* o_part, float* lse_part,
                       unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_tmap_3d(&mq, q, s.d, s.hq, s.T, 64, s.G, 1, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&mk, k, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&mv, v, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  FwdArgs a{cu_seqlens, cu_blocks, row_ptr, ent,   s.ndoc, s.T,   s.hq,
            s.hkv,      s.K,       s.nb_bound, s.softmax_scale, o_part, lse_part, status};
  return s.d == 128 ? launch_fwd_d<128>(s, mq, mk, mv, a, st)
                    : launch_fwd_d<64>(s, mq, mk, mv, a, st);
}

}  // namespace msa
